// tmap.h -- TMA tensor maps for batched row-major matrices.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace dion {

enum class TmapType { BF16, F32 };

// A [batch][rows][inner] tensor with the given pitches; boxes of
// box_rows x box_inner elements land in shared memory with the 128-byte
// swizzle.  Out-of-range elements read as zero.  Returns false if the driver
// entry point is missing or an alignment rule is broken (base, pitches 16-byte
// aligned; box_inner * element size a multiple of 16 and at most 128 bytes).
bool make_tmap_3d(CUtensorMap* out, const void* base, TmapType type, uint64_t inner, uint64_t rows, uint64_t batch,
                  uint64_t row_pitch_bytes, uint64_t batch_pitch_bytes, uint32_t box_inner, uint32_t box_rows);

// The same with the 64-byte swizzle (box_inner * element size at most 64
// bytes): 16-byte chunk c of box row r lands at r * rowbytes + 16 (c ^ ((r / 2) % 4))
// for 64-byte rows.
bool make_tmap_3d_sw64(CUtensorMap* out, const void* base, TmapType type, uint64_t inner, uint64_t rows,
                       uint64_t batch, uint64_t row_pitch_bytes, uint64_t batch_pitch_bytes, uint32_t box_inner,
                       uint32_t box_rows);

}  // namespace dion
