// api.cu -- the C ABI of libdion: argument checks, workspace layout, dispatch.
#include <algorithm>
#include <cmath>

#include "internal.h"

namespace dion {

static size_t carve(size_t& off, size_t bytes)
{
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
}

// Splits of a streaming contraction so that one wave of CTAs covers the SMs
// (one CTA per SM) of the current device; fixed per shape and device, so
// that the workspace size is too.
static int stream_splits(long long base_ctas, int kchunks)
{
    const int sms = num_sms();
    int s = (int)((sms + base_ctas / 2) / base_ctas);
    if (s < 1) s = 1;
    if (s > kchunks) s = kchunks;
    const int per = (kchunks + s - 1) / s;
    return (kchunks + per - 1) / per;
}

DionLayout dion_layout(int batch, int m, int n, int r, dion_dtype dt)
{
    DionLayout L{};
    L.tc = (dt == DION_BF16);
    L.rp = L.tc ? (int)align_up((size_t)r, 64) : r;   // MN-major operand blocks are 64 wide
    const size_t b = (size_t)batch, f = sizeof(float), h = 2, rp = (size_t)L.rp;
    L.ksplit = L.ksplit_r = 1;
    size_t off = 0;
    L.status = carve(off, 256);
    L.P0 = carve(off, b * m * rp * f);
    L.P1 = carve(off, b * m * rp * f);
    L.R = carve(off, b * n * rp * f);
    const size_t nb8 = (size_t)(r + 7) / 8;
    L.S = carve(off, b * std::max((size_t)r * r, nb8 * (nb8 + 1) / 2 * 64) * f);   // also the block-major Gram
    L.W = carve(off, b * r * r * f);
    L.dead = carve(off, b * r * sizeof(int));
    L.inv = carve(off, b * rp * f);
    L.hard = carve(off, (b + 1) * sizeof(int));
    if (L.tc) {
        const int rch = (int)cdiv(L.rp, 256);
        // wider than one 256-column chunk: B = M + G is formed once in bf16
        // (row-major and transposed) and both products run as TMA GEMMs
        L.wide = rch > 1;
        L.ksplit = L.wide ? 1 : stream_splits(cdiv(m, 128) * rch * batch, (int)cdiv(n, 64));
        L.ksplit_r = L.wide ? 1 : stream_splits(cdiv(n, 128) * rch * batch, (int)cdiv(m, 64));
        const size_t rows = std::max((size_t)L.ksplit * m, (size_t)L.ksplit_r * n);
        L.Ppart = carve(off, rows * b * rp * f);
        L.Qt16 = carve(off, b * rp * align_up((size_t)n, 8) * h);
        L.P16 = carve(off, b * m * rp * h);
        L.R16 = carve(off, b * n * rp * h);
        L.Q16 = carve(off, b * n * rp * h);
        L.P3 = carve(off, 3 * b * m * rp * h);
        L.P3b = carve(off, 3 * b * m * rp * h);
        L.Z3 = carve(off, 3 * b * r * rp * h);
        L.S6 = carve(off, 6 * b * r * r * f);
        L.normp = carve(off, b * (size_t)cdiv(n, 32) * rp * f);
        L.rcount = carve(off, b * sizeof(int));
        L.emax = carve(off, b * sizeof(int));
        if (L.wide) {   // bf16 B, read K-major by B Q and MN-major by B^T P
            const size_t np = align_up((size_t)n, 8);
            L.B16 = carve(off, b * m * np * h);
        } else if (n % 8 == 0) {   // the B Q pass stores B = M + G in bf16 for the B^T P GEMM
            L.b16_narrow = true;
            L.B16 = carve(off, b * m * (size_t)n * h);
        } else {
            L.B16 = off;
        }
        L.S64 = L.S6;   // 6 b r r floats hold the 2 b r r doubles of the float64 first pass
        L.nbc = chol_block_size(r);
        if (L.nbc > 0) {
            const size_t nb = (size_t)L.nbc;
            L.ZJ = carve(off, 3 * b * nb * nb * h);
            L.A3 = carve(off, 3 * b * r * nb * h);
        } else {
            L.ZJ = L.A3 = off;
        }
    } else {
        L.nbc = 0;
        L.wide = false;
        L.ZJ = L.A3 = L.B16 = off;
        L.Ppart = L.Qt16 = L.P16 = L.R16 = L.Q16 = off;
        L.P3 = L.P3b = L.Z3 = L.S6 = L.normp = L.rcount = L.emax = off;
        L.S64 = carve(off, 2 * b * r * r * sizeof(double));
    }
    L.total = off;
    return L;
}

MuonLayout muon_layout(int batch, int m, int n, int head_dim, dion_dtype dt)
{
    MuonLayout L{};
    L.hd = head_dim > 0 ? head_dim : n;
    L.heads = n / L.hd;
    L.nb = batch * L.heads;
    L.tr = m > L.hd;
    L.s = std::min(m, L.hd);
    L.l = std::max(m, L.hd);
    L.tc = (dt == DION_BF16);
    const size_t nb = (size_t)L.nb, f = sizeof(float);
    size_t off = 0;
    L.status = carve(off, 256);
    L.nrm = carve(off, nb * f);
    if (L.tc) {
        L.lp = (int)align_up((size_t)L.l, 8);
        L.sp = (int)align_up((size_t)L.s, 8);
        const size_t h = sizeof(uint16_t);
        L.Xa = carve(off, nb * L.s * L.lp * h);
        L.Xb = carve(off, nb * L.s * L.lp * h);
        L.XTa = L.XTb = off;   // no transposed copy: Bm Y reads Y MN-major
        L.A = carve(off, nb * L.s * L.sp * h);
        L.Bm = carve(off, nb * L.s * L.sp * h);
    } else {
        L.lp = L.l;
        L.sp = L.s;
        const size_t sl = (size_t)L.s * L.l, ss = (size_t)L.s * L.s;
        L.Xa = carve(off, nb * sl * f);
        L.Xb = carve(off, nb * sl * f);
        L.XTa = L.XTb = off;
        L.A = carve(off, nb * ss * f);
        L.Bm = carve(off, nb * ss * f);
    }
    L.total = off;
    return L;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace dion

using namespace dion;

extern "C" const char* dion_status_string(dion_status s)
{
    switch (s) {
    case DION_OK: return "ok";
    case DION_ERR_INVALID_ARG: return "invalid argument";
    case DION_ERR_UNSUPPORTED: return "unsupported";
    case DION_ERR_WORKSPACE: return "workspace missing or too small";
    case DION_ERR_CUDA: return "CUDA error";
    case DION_ERR_NUMERIC: return "numeric breakdown on the device";
    }
    return "unknown status";
}

static bool dion_shape_ok(int batch, int m, int n, int r, dion_dtype dt)
{
    return batch >= 1 && batch <= 65535 && m >= 1 && n >= 1 && r >= 1 && r <= std::min(m, n) &&
           (dt == DION_F32 || dt == DION_BF16);
}

extern "C" dion_status dion_workspace_size(int batch, int m, int n, int r, dion_dtype dt, size_t* bytes)
{
    if (!bytes || !dion_shape_ok(batch, m, n, r, dt)) return DION_ERR_INVALID_ARG;
    *bytes = dion_layout(batch, m, n, r, dt).total;
    return DION_OK;
}

extern "C" dion_status dion_workspace_panels(int batch, int m, int n, int r, dion_dtype dt, size_t* p_offset,
                                             int* p_ld, size_t* r_offset, int* r_ld)
{
    if (!dion_shape_ok(batch, m, n, r, dt)) return DION_ERR_INVALID_ARG;
    const DionLayout L = dion_layout(batch, m, n, r, dt);
    if (p_offset) *p_offset = L.P0;
    if (p_ld) *p_ld = L.rp;
    if (r_offset) *r_offset = L.R;
    if (r_ld) *r_ld = L.rp;
    return DION_OK;
}

static dion_status dion_step_any(int batch, int m, int n, int r, dion_dtype dt, void* X, const void* G, float* M,
                                 float* Q, float mu, float lr, float weight_decay, const float* hyper, void* workspace,
                                 size_t workspace_bytes, void* cuda_stream)
{
    if (!dion_shape_ok(batch, m, n, r, dt)) return DION_ERR_INVALID_ARG;
    if (!X || !G || !M || !Q) return DION_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(G) || !aligned16(M) || !aligned16(Q)) return DION_ERR_INVALID_ARG;
    if (!std::isfinite(mu) || !std::isfinite(lr) || !std::isfinite(weight_decay)) return DION_ERR_INVALID_ARG;
    const DionLayout L = dion_layout(batch, m, n, r, dt);
    // the tensor-core path addresses the batch x n x rp panel of R in 4-column units with 32-bit indices
    if (L.tc && (long long)batch * n * (L.rp / 4) >= (1ll << 31)) return DION_ERR_UNSUPPORTED;
    if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < L.total) return DION_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    if (L.tc) return dion_step_tc(batch, m, n, r, X, G, M, Q, mu, lr, weight_decay, hyper, (char*)workspace, L, st);
    return dion_step_simt(batch, m, n, r, dt, X, G, M, Q, mu, lr, weight_decay, hyper, (char*)workspace, L, st);
}

extern "C" dion_status dion_step_batched(int batch, int m, int n, int r, dion_dtype dt, void* X, const void* G,
                                         float* M, float* Q, float mu, float lr, float weight_decay,
                                         void* workspace, size_t workspace_bytes, void* cuda_stream)
{
    return dion_step_any(batch, m, n, r, dt, X, G, M, Q, mu, lr, weight_decay, nullptr, workspace, workspace_bytes,
                         cuda_stream);
}

extern "C" dion_status dion_step_batched_dev(int batch, int m, int n, int r, dion_dtype dt, void* X, const void* G,
                                             float* M, float* Q, const float* hyper, void* workspace,
                                             size_t workspace_bytes, void* cuda_stream)
{
    if (!hyper || ((uintptr_t)hyper & 3u)) return DION_ERR_INVALID_ARG;
    return dion_step_any(batch, m, n, r, dt, X, G, M, Q, 0.f, 0.f, 0.f, hyper, workspace, workspace_bytes,
                         cuda_stream);
}

static bool muon_shape_ok(int batch, int m, int n, int head_dim, dion_dtype dt)
{
    if (batch < 1 || m < 1 || n < 1 || head_dim < 0) return false;
    if (head_dim > 0 && n % head_dim != 0) return false;
    if (dt != DION_F32 && dt != DION_BF16) return false;
    const long long nb = (long long)batch * (head_dim > 0 ? n / head_dim : 1);
    return nb <= 65535;
}

extern "C" dion_status muon_workspace_size(int batch, int m, int n, int head_dim, dion_dtype dt, size_t* bytes)
{
    if (!bytes || !muon_shape_ok(batch, m, n, head_dim, dt)) return DION_ERR_INVALID_ARG;
    *bytes = muon_layout(batch, m, n, head_dim, dt).total;
    return DION_OK;
}

extern "C" dion_status muon_ns_batched(int batch, int m, int n, int head_dim, dion_dtype dt, void* X, const void* G,
                                       float* M, void* O, int steps, const float* coeff, float mu, float lr,
                                       float weight_decay, void* workspace, size_t workspace_bytes,
                                       void* cuda_stream)
{
    if (!muon_shape_ok(batch, m, n, head_dim, dt)) return DION_ERR_INVALID_ARG;
    if (!G || (!X && !O) || !coeff || steps < 0) return DION_ERR_INVALID_ARG;
    if (!aligned16(G) || (X && !aligned16(X)) || (M && !aligned16(M)) || (O && !aligned16(O)))
        return DION_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
        if (!std::isfinite(coeff[i])) return DION_ERR_INVALID_ARG;
    if (!std::isfinite(mu) || !std::isfinite(lr) || !std::isfinite(weight_decay)) return DION_ERR_INVALID_ARG;
    const MuonLayout L = muon_layout(batch, m, n, head_dim, dt);
    if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < L.total) return DION_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    if (L.tc)
        return muon_tc(batch, m, n, dt, X, G, M, O, steps, coeff, mu, lr, weight_decay, (char*)workspace, L, st);
    return muon_simt(batch, m, n, dt, X, G, M, O, steps, coeff, mu, lr, weight_decay, (char*)workspace, L, st);
}

extern "C" dion_status dion_get_status(const void* workspace, int* device_status)
{
    if (!workspace || !device_status) return DION_ERR_INVALID_ARG;
    int v = 0;
    if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DION_ERR_CUDA;
    *device_status = v;
    return v ? DION_ERR_NUMERIC : DION_OK;
}
