// tmap.cu -- host-side TMA tensor-map encoding (driver entry point fetched
// through the runtime, so libdion needs no link against libcuda).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tmap.h"

namespace dion {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    // looked up once, thread-safely (function-local static initialization)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000)p;
        return nullptr;
    }();
    return fn;
}

static bool encode_3d(CUtensorMap* out, const void* base, TmapType type, uint64_t inner, uint64_t rows,
                      uint64_t batch, uint64_t row_pitch_bytes, uint64_t batch_pitch_bytes, uint32_t box_inner,
                      uint32_t box_rows, CUtensorMapSwizzle swizzle, uint32_t span)
{
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const uint32_t esize = (type == TmapType::BF16) ? 2u : 4u;
    if (((uintptr_t)base & 15u) || (row_pitch_bytes & 15u) || (batch_pitch_bytes & 15u)) return false;
    if ((box_inner * esize) % 16u || box_inner * esize > span || box_rows == 0 || box_rows > 256u) return false;
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {row_pitch_bytes, batch_pitch_bytes};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(out, type == TmapType::BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap* out, const void* base, TmapType type, uint64_t inner, uint64_t rows, uint64_t batch,
                  uint64_t row_pitch_bytes, uint64_t batch_pitch_bytes, uint32_t box_inner, uint32_t box_rows)
{
    return encode_3d(out, base, type, inner, rows, batch, row_pitch_bytes, batch_pitch_bytes, box_inner, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B, 128u);
}

bool make_tmap_3d_sw64(CUtensorMap* out, const void* base, TmapType type, uint64_t inner, uint64_t rows,
                       uint64_t batch, uint64_t row_pitch_bytes, uint64_t batch_pitch_bytes, uint32_t box_inner,
                       uint32_t box_rows)
{
    return encode_3d(out, base, type, inner, rows, batch, row_pitch_bytes, batch_pitch_bytes, box_inner, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_64B, 64u);
}

}  // namespace dion
