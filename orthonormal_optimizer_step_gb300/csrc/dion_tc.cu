// dion_tc.cu -- the Dion step on the tensor cores, for bf16 weights/gradients.
//
// Per megabatch of m x n matrices at rank r (rp = r rounded up to 64, the
// width of one 128-byte swizzle block of bf16):
//   1. dion_prep_qt  : Qt = bf16(Q^T)                      (rp x n, K-major operand)
//   2. dion_bq_tc    : P = B Q with B = M + G formed in registers, rounded to
//                      bf16 and written straight into the swizzled MMA operand
//                      tile (B is never stored); split over n, fp32 partials
//   3-5. CholeskyQR2 of P (float32 accuracy; products on the tensor cores,
//      qr_tc.cu): its first pass reads the partials, its last product also
//      writes P16 = bf16(P)
//   6. dion_btp_tc   : R = B^T P, contracting over m: both operands are read
//                      MN-major (B rows are K rows), so B is again formed in
//                      registers without any transpose; split over m
//   7. dion_rsum     : R = sum of partials, R16 = bf16(R), column norms (the
//                      last CTA of each matrix finishes them)
//   8. dion_qemit    : Q = R / ||R_j|| (caller's fp32 Q) and Q16
//   9. dion_update_tc: per 128 x 64 tile, two accumulators P R^T and P Q^T in
//                      tensor memory; the epilogue streams M, G, X once:
//                      M <- M + G - (1-mu) P R^T,  X <- (1-lr wd) X - lr sqrt(m/n) P Q^T
// The MMAs are tcgen05.mma kind::f16 (bf16 in, fp32 accumulate); tiles reach
// shared memory by TMA (Q, P, R operands) or from the producer warps (B).
#include "internal.h"
#include "tc.cuh"
#include "tc_gemm.cuh"
#include "tmap.h"

namespace dion {

int num_sms();

namespace {

constexpr int kBM = 128, kBK = 64;

__device__ __forceinline__ uint4 pack8(const float (&v)[8])
{
    uint4 u;
    u.x = tc::pack_bf16x2(v[0], v[1]);
    u.y = tc::pack_bf16x2(v[2], v[3]);
    u.z = tc::pack_bf16x2(v[4], v[5]);
    u.w = tc::pack_bf16x2(v[6], v[7]);
    return u;
}

// v[0..8) = M[o..o+8) + G[o..o+8) for columns col..col+7 of row i; zero outside
// the matrix.  VEC: 16-byte vector loads (needs n % 8 == 0).
template <bool VEC>
__device__ __forceinline__ void load_b8(const float* M, const bf16* G, long long rowbase, int i, int m, int col, int n,
                                        float (&v)[8])
{
    if (VEC && i < m && col + 8 <= n) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(M + rowbase + col));
        const float4 c = __ldg(reinterpret_cast<const float4*>(M + rowbase + col + 4));
        const uint4 g = __ldg(reinterpret_cast<const uint4*>(G + rowbase + col));
        const bf16* h = reinterpret_cast<const bf16*>(&g);
        v[0] = a.x + __bfloat162float(h[0]); v[1] = a.y + __bfloat162float(h[1]);
        v[2] = a.z + __bfloat162float(h[2]); v[3] = a.w + __bfloat162float(h[3]);
        v[4] = c.x + __bfloat162float(h[4]); v[5] = c.y + __bfloat162float(h[5]);
        v[6] = c.z + __bfloat162float(h[6]); v[7] = c.w + __bfloat162float(h[7]);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = col + e;
            v[e] = (i < m && c < n) ? M[rowbase + c] + __bfloat162float(G[rowbase + c]) : 0.f;
        }
    }
}

// Raw loads of 8 consecutive elements of M and G (issued early, converted later).
struct Raw8 {
    float4 a, c;
    uint4 g;
};

template <bool VEC>
__device__ __forceinline__ void fetch_b8(const float* M, const bf16* G, long long rowbase, int i, int m, int col, int n,
                                         Raw8& r)
{
    if (VEC && i < m && col + 8 <= n) {
        r.a = __ldg(reinterpret_cast<const float4*>(M + rowbase + col));
        r.c = __ldg(reinterpret_cast<const float4*>(M + rowbase + col + 4));
        r.g = __ldg(reinterpret_cast<const uint4*>(G + rowbase + col));
    } else {
        float v[8];
        load_b8<false>(M, G, rowbase, i, m, col, n, v);   // already summed; G part set to zero
        r.a = make_float4(v[0], v[1], v[2], v[3]);
        r.c = make_float4(v[4], v[5], v[6], v[7]);
        r.g = make_uint4(0u, 0u, 0u, 0u);
    }
}

__device__ __forceinline__ uint4 sum_pack8(const Raw8& r)
{
    const bf16* h = reinterpret_cast<const bf16*>(&r.g);
    float v[8] = {r.a.x + __bfloat162float(h[0]), r.a.y + __bfloat162float(h[1]), r.a.z + __bfloat162float(h[2]),
                  r.a.w + __bfloat162float(h[3]), r.c.x + __bfloat162float(h[4]), r.c.y + __bfloat162float(h[5]),
                  r.c.z + __bfloat162float(h[6]), r.c.w + __bfloat162float(h[7])};
    return pack8(v);
}

struct PassArgs {
    int m, n, rp, batch;
    int splits;             // K splits (fp32 partial planes)
    int kchunks_per_split;  // 64-wide K chunks per split
    int kchunks;            // total K chunks
    const float* M;
    const bf16* G;
    float* part;            // [split][batch][rows][rp] fp32 partial products
    int* status;
    bool store_b;           // B Q pass only: also store B = M + G, as rounded for the MMA, through tmS
    // B Q pass with one split only, if P3 is set: the epilogue writes the
    // three bf16 terms of P (term t of matrix b at P3 + (3 b + t) m rp, the
    // first CholeskyQR pass's input) instead of the float32 partial, and P
    // itself as float32 to Pf when set (the blocked factorization's input)
    bf16* P3;
    float* Pf;
};

constexpr int kProducers = 512;                  // warps 0..15 build the B tiles
constexpr int kMmaWarp = kProducers / 32;        // warp 16 issues the MMAs
constexpr int kEpiWarp0 = kMmaWarp + 1;          // warps 17..20 drain the accumulators
constexpr int kPassWarps = kEpiWarp0 + 4;
constexpr int kPerProducer = 1024 / kProducers;  // 8-element groups of a 128 x 64 tile per producer thread
constexpr int kStages = 4;
constexpr uint32_t kAB = kBM * kBK * 2;          // 16 KB bf16 A tile
constexpr uint32_t kBB = 256 * kBK * 2;          // up to 32 KB B tile
constexpr uint32_t kStage = kAB + kBB;
constexpr size_t kPassSmem = (size_t)kStages * kStage + 1024 + 256;

// The two streaming passes (rp <= 256; wider ranks use the TMA GEMMs), as a
// persistent kernel over work units (batch entry, K split, 128-row output
// tile; tiles fastest, so concurrent CTAs share the operand chunks in L2).
// MN_A = false: P = B Q, A tile = 128 rows of B x 64 columns, K-major.
// MN_A = true:  R = B^T P, A tile = 64 rows of B x 128 columns, MN-major.
// The other operand (Q16 or P16, row-major K x rp) is MN-major in both.
// Producer warps form B = M + G in registers (two chunks of loads in flight,
// across unit boundaries), round to bf16 and write the swizzled A tile; one
// thread adds the operand tile (Q^T or P) by TMA.  The accumulator is double
// buffered in tensor memory, so the epilogue warps write the fp32 partials of
// one unit while the next unit streams.
template <bool MN_A, bool VEC>
__global__ void __launch_bounds__(kPassWarps * 32, 1) dion_pass_kernel(const __grid_constant__ CUtensorMap tmB,
                                                                       const __grid_constant__ CUtensorMap tmS,
                                                                       PassArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(smem + kStages * kStage);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = (uint32_t*)(acc_empty + 2);
    int* abort_flag = (int*)(tmem_slot + 1);
    volatile int* abrt = abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int out_rows = MN_A ? a.n : a.m;
    const int tiles = (out_rows + kBM - 1) / kBM;
    const int units = tiles * a.splits * a.batch;
    const int nN = a.rp;                               // MMA N (multiple of 64, at most 256)
    const uint32_t b_bytes = (uint32_t)(nN / 64) * 8192u;   // B operand: nN/64 MN-major 64 x 64 boxes
    auto unit_of = [&](int u, int& b, int& split, int& tile, int& kc0, int& nk) {
        tile = u % tiles;
        split = (u / tiles) % a.splits;
        b = u / (tiles * a.splits);
        kc0 = split * a.kchunks_per_split;
        nk = min(a.kchunks_per_split, a.kchunks - kc0);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], kProducers / 32 + 1);   // one arrive per producer warp + the TMA
            tc::mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&acc_full[s], 1);
            tc::mbar_init(&acc_empty[s], 4);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kMmaWarp) {
        // ---------------- producers: B = M + G -> bf16 -> swizzled A tile
        Raw8 cur[kPerProducer], nxt[kPerProducer];
        uint32_t off[kPerProducer];
        auto fetch = [&](int b, int tile, int kc, Raw8 (&dst)[kPerProducer]) {
            const int k0 = kc * kBK;
#pragma unroll
            for (int v = 0; v < kPerProducer; ++v) {
                const int g = threadIdx.x + kProducers * v;
                if (!MN_A) {
                    const int row = g >> 3, ch = g & 7;             // 128 rows x 8 chunks
                    const int i = tile * kBM + row;
                    fetch_b8<VEC>(a.M, a.G, ((long long)b * a.m + i) * a.n, i, a.m, k0 + ch * 8, a.n, dst[v]);
                    off[v] = tc::sw128_offset(row, ch);
                } else {
                    const int row = g >> 4, ch = g & 15;            // 64 K-rows x 16 chunks
                    const int i = k0 + row;
                    fetch_b8<VEC>(a.M, a.G, ((long long)b * a.m + i) * a.n, i, a.m, tile * kBM + ch * 8, a.n,
                                  dst[v]);
                    off[v] = (ch >> 3) * 8192u + tc::sw128_offset(row, ch & 7);
                }
            }
        };
        // cursor over the flattened (unit, chunk) sequence of this CTA
        int u = blockIdx.x, b = 0, split = 0, tile = 0, kc0 = 0, nk = 0, kc = 0;
        if (u < units) unit_of(u, b, split, tile, kc0, nk);
        int nu = u, nb = b, ntile = tile, nkc0 = kc0, nnk = nk, nkc = 0;   // the chunk after the current one
        auto advance = [&]() {
            if (++nkc >= nnk) {
                nu += gridDim.x;
                nkc = 0;
                int sp;
                if (nu < units) unit_of(nu, nb, sp, ntile, nkc0, nnk);
            }
        };
        if (u < units) fetch(b, tile, kc0, cur);
        advance();
        int stage = 0;
        uint32_t ph = 0;
        while (u < units && !*abrt) {
            if (nu < units) fetch(nb, ntile, nkc0 + nkc, nxt);
            if (lane == 0) tc::mbar_wait(&empty[stage], ph ^ 1, abrt, a.status);
            __syncwarp();
            if (*abrt) break;
            uint8_t* sA = smem + stage * kStage;
            const int k0 = (kc0 + kc) * kBK;
            if (threadIdx.x == 0) {
                tc::mbar_arrive_expect_tx(&full[stage], b_bytes);
                for (int blk = 0; blk * 64 < nN; ++blk)
                    tc::tma_load_3d(sA + kAB + blk * 8192, &tmB, &full[stage], blk * 64, k0, b);
            }
#pragma unroll
            for (int v = 0; v < kPerProducer; ++v) *reinterpret_cast<uint4*>(sA + off[v]) = sum_pack8(cur[v]);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&full[stage]);
            if (++stage == kStages) { stage = 0; ph ^= 1; }
#pragma unroll
            for (int v = 0; v < kPerProducer; ++v) cur[v] = nxt[v];
            u = nu; b = nb; tile = ntile; kc0 = nkc0; nk = nnk; kc = nkc;
            advance();
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc = tc::make_idesc(kBM, nN, 1, MN_A, true);
            int stage = 0, it = 0;
            uint32_t ph = 0;
            int pend = -1;   // stage whose release waits for its B store to finish reading it
            for (int u = blockIdx.x; u < units && !*abrt; u += gridDim.x, ++it) {
                int b, split, tile, kc0, nk;
                unit_of(u, b, split, tile, kc0, nk);
                const int buf = it & 1;
                if (!tc::mbar_wait(&acc_empty[buf], ((it >> 1) & 1) ^ 1, abrt, a.status)) break;
                tc::tc_fence_after();
                const uint32_t d = tmem + buf * 256;
                bool ok = true;
                for (int kc = 0; kc < nk; ++kc) {
                    if (!tc::mbar_wait(&full[stage], ph, abrt, a.status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(smem + stage * kStage), b0 = a0 + kAB;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t ad = MN_A ? tc::make_sdesc(a0 + k * 2048, 8192, 1024)
                                                 : tc::make_sdesc(a0 + k * 32, 16, 1024);
                        const uint64_t bd = tc::make_sdesc(b0 + k * 2048, 8192, 1024);
                        tc::mma_bf16(d, ad, bd, idesc, (kc | k) != 0);
                    }
                    if (!MN_A && a.store_b) {
                        // the bf16 B tile (128 rows x 64 columns, 128-byte swizzled as the
                        // tensor map expects) to global memory for the B^T P GEMM.  A stage
                        // is released only after its store has read it; the store of this
                        // chunk stays in flight and releases its stage one chunk later
                        tc::tma_store_3d(&tmS, smem + stage * kStage, (kc0 + kc) * kBK, tile * kBM, b);
                        tc::tma_store_commit();
                        if (pend >= 0) {
                            tc::tma_store_wait_read1();
                            tc::mma_commit(&empty[pend]);
                        }
                        pend = stage;
                    } else {
                        tc::mma_commit(&empty[stage]);
                    }
                    if (++stage == kStages) { stage = 0; ph ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit(&acc_full[buf]);
            }
            if (!MN_A && a.store_b) {
                if (pend >= 0) {
                    tc::tma_store_wait_read();
                    tc::mma_commit(&empty[pend]);
                }
                tc::tma_store_wait_all();
            }
        }
    } else {
        // ---------------- epilogue: TMEM -> fp32 partials
        const int q = warp & 3;                        // TMEM lane quarter of this warp
        int it = 0;
        for (int u = blockIdx.x; u < units && !*abrt; u += gridDim.x, ++it) {
            int b, split, tile, kc0, nk;
            unit_of(u, b, split, tile, kc0, nk);
            const int buf = it & 1;
            if (!tc::mbar_wait(&acc_full[buf], (it >> 1) & 1, abrt, a.status)) break;
            tc::tc_fence_after();
            const int row = tile * kBM + q * 32 + lane;
            float* out = a.part + (((long long)split * a.batch + b) * out_rows + row) * a.rp;
            const long long pn = (long long)a.m * a.rp, po = (long long)row * a.rp;
            for (int c0 = 0; c0 < nN; c0 += 32) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 256 + c0), v);
                tc::tmem_ld_wait();
                if (row < out_rows) {
                    if (!MN_A && a.P3) {
                        // the split of P into three bf16 terms (24 significant bits), columns
                        // past r are zero already (so are those of Q)
                        bf16* t0 = a.P3 + 3ll * b * pn + po + c0;
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            uint32_t w[3][2];
#pragma unroll
                            for (int h = 0; h < 4; h += 2) {
                                uint32_t p1 = 0, p2 = 0, p3 = 0;
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const float x = __uint_as_float(v[j + h + e]);
                                    const bf16 h1 = __float2bfloat16_rn(x);
                                    const float r1 = x - __bfloat162float(h1);
                                    const bf16 h2 = __float2bfloat16_rn(r1);
                                    const bf16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
                                    p1 |= (uint32_t)__bfloat16_as_ushort(h1) << (16 * e);
                                    p2 |= (uint32_t)__bfloat16_as_ushort(h2) << (16 * e);
                                    p3 |= (uint32_t)__bfloat16_as_ushort(h3) << (16 * e);
                                }
                                w[0][h / 2] = p1;
                                w[1][h / 2] = p2;
                                w[2][h / 2] = p3;
                            }
#pragma unroll
                            for (int t = 0; t < 3; ++t)
                                *reinterpret_cast<uint2*>(t0 + t * pn + j) = make_uint2(w[t][0], w[t][1]);
                        }
                        if (a.Pf) {
                            float* pf = a.Pf + (long long)b * pn + po + c0;
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                *reinterpret_cast<float4*>(pf + j) =
                                    make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(out + c0 + j) =
                                make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                            __uint_as_float(v[j + 3]));
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
        }
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------ the update pass
struct UpdArgs {
    int m, n, rp, kchunks;
    float* M;
    const bf16* G;
    bf16* X;
    StepHyper hp;
    int* status;
};

constexpr int kUBN = 64, kUStages = 3;
constexpr uint32_t kUA = kBM * kBK * 2, kUB = kUBN * kBK * 2, kUStage = kUA + 2 * kUB;
constexpr size_t kUpdSmem = (size_t)kUStages * kUStage + 1024 + 256;

template <bool VEC>
__global__ void __launch_bounds__(192) dion_update_tc_kernel(const __grid_constant__ CUtensorMap tmP,
                                                             const __grid_constant__ CUtensorMap tmR,
                                                             const __grid_constant__ CUtensorMap tmQ, UpdArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(smem + kUStages * kUStage);
    uint64_t* empty = full + kUStages;
    uint64_t* done = empty + kUStages;
    uint32_t* tmem_slot = (uint32_t*)(done + 1);
    int* abort_flag = (int*)(tmem_slot + 1);
    volatile int* abrt = abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float one_minus_mu, decay, scale;
    a.hp.get(one_minus_mu, decay, scale);
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0 && !a.hp.finite())
        atomicOr(a.status, kStatusNonFinite);
    const int nt = blockIdx.x, mt = blockIdx.y, b = blockIdx.z;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kUStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(done, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 5) {
        tc::tmem_alloc(tmem_slot, 128);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        if (lane == 0) {
            for (int kc = 0; kc < a.kchunks; ++kc) {
                const int stage = kc % kUStages;
                const uint32_t ph = (kc / kUStages) & 1;
                if (!tc::mbar_wait(&empty[stage], ph ^ 1, abrt, a.status)) break;
                uint8_t* s = smem + stage * kUStage;
                tc::mbar_arrive_expect_tx(&full[stage], kUStage);
                tc::tma_load_3d(s, &tmP, &full[stage], kc * kBK, mt * kBM, b);
                tc::tma_load_3d(s + kUA, &tmR, &full[stage], kc * kBK, nt * kUBN, b);
                tc::tma_load_3d(s + kUA + kUB, &tmQ, &full[stage], kc * kBK, nt * kUBN, b);
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            const uint32_t idesc = tc::make_idesc(kBM, kUBN, 1, false, false);
            for (int kc = 0; kc < a.kchunks; ++kc) {
                const int stage = kc % kUStages;
                const uint32_t ph = (kc / kUStages) & 1;
                if (!tc::mbar_wait(&full[stage], ph, abrt, a.status)) break;
                tc::tc_fence_after();
                const uint32_t a0 = tc::smem_u32(smem + stage * kUStage), r0 = a0 + kUA, q0 = r0 + kUB;
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) {
                    const uint64_t ad = tc::make_sdesc(a0 + k * 32, 16, 1024);
                    tc::mma_bf16(tmem, ad, tc::make_sdesc(r0 + k * 32, 16, 1024), idesc, (kc | k) != 0);
                    tc::mma_bf16(tmem + kUBN, ad, tc::make_sdesc(q0 + k * 32, 16, 1024), idesc, (kc | k) != 0);
                }
                tc::mma_commit(&empty[stage]);
            }
            tc::mma_commit(done);
        }
    } else {
        // epilogue warps 0..3: row = one TMEM lane
        const int i = mt * kBM + warp * 32 + lane;
        const bool ok = tc::mbar_wait(done, 0, abrt, a.status);
        tc::tc_fence_after();
        for (int c0 = 0; c0 < kUBN; c0 += 32) {
            uint32_t pr[32], pq[32];
            tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, pr);
            tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(kUBN + c0), pq);
            tc::tmem_ld_wait();
            const int j0 = nt * kUBN + c0;
            if (!ok || i >= a.m || j0 >= a.n) continue;
            const long long o = ((long long)b * a.m + i) * a.n + j0;
            if (VEC && j0 + 32 <= a.n) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float4 m0 = *reinterpret_cast<const float4*>(a.M + o + 8 * q);
                    float4 m1 = *reinterpret_cast<const float4*>(a.M + o + 8 * q + 4);
                    const uint4 g = __ldg(reinterpret_cast<const uint4*>(a.G + o + 8 * q));
                    const uint4 x = *reinterpret_cast<const uint4*>(a.X + o + 8 * q);
                    const bf16* gh = reinterpret_cast<const bf16*>(&g);
                    const bf16* xh = reinterpret_cast<const bf16*>(&x);
                    float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
                    float xv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        mv[e] = mv[e] + __bfloat162float(gh[e]) - one_minus_mu * __uint_as_float(pr[8 * q + e]);
                        xv[e] = decay * __bfloat162float(xh[e]) - scale * __uint_as_float(pq[8 * q + e]);
                    }
                    *reinterpret_cast<float4*>(a.M + o + 8 * q) = make_float4(mv[0], mv[1], mv[2], mv[3]);
                    *reinterpret_cast<float4*>(a.M + o + 8 * q + 4) = make_float4(mv[4], mv[5], mv[6], mv[7]);
                    *reinterpret_cast<uint4*>(a.X + o + 8 * q) = pack8(xv);
                }
            } else {
                const int nv = min(32, a.n - j0);
                for (int e = 0; e < nv; ++e) {
                    a.M[o + e] = a.M[o + e] + __bfloat162float(a.G[o + e]) - one_minus_mu * __uint_as_float(pr[e]);
                    a.X[o + e] = __float2bfloat16_rn(decay * __bfloat162float(a.X[o + e]) -
                                                     scale * __uint_as_float(pq[e]));
                }
            }
        }
        tc::tc_fence_before();
    }
    __syncthreads();
    if (warp == 5) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 128);
    }
}

// ------------------------------------------------ persistent update pass
// One CTA per SM walks the 128 x 64 tiles of M and X.  The M, G and X tiles
// move between HBM and shared memory by TMA (two tile buffers, so the loads
// of the next tile run under the math and the stores of this one), the P, R
// and Q operands stream through two K stages, and the two accumulators
// (P R^T, P Q^T) are double-buffered in tensor memory.
//   warps 0..7: epilogue (warp w: TMEM lane quarter w % 4, 32-column half w / 4;
//               two warps per scheduler, so the TMEM and shared-memory
//               latencies of one overlap the arithmetic of the other)
//   warp 8: TMA producer     warp 9: MMA issuer
struct UpdPArgs {
    int m, n, batch, kchunks, tiles_m, tiles_n;
    StepHyper hp;
    int* status;
    // tile order within a matrix: m_fast walks the row tiles fastest (the P
    // panel cycles, each R/Q chunk is used by consecutive tiles), else the
    // column tiles (R/Q cycle, each P chunk is used by consecutive tiles).
    // The shorter direction goes fastest, so the operands that cycle stay a
    // few MB and remain in L2 while M, G and X stream through it.
    int m_fast;
};

constexpr uint32_t kPStage = kUStage;                              // 32 KB of operands per K chunk
constexpr uint32_t kEM = 2 * 16384, kEG = 16384, kEX = 16384;      // M (two 32-column boxes), G, X
constexpr uint32_t kEBuf = kEM + kEG + kEX;                        // 64 KB
// Ring depths of the persistent update: operand stages per K chunk and M/G/X
// tile buffers.  Short K ranges (rp <= 256) double-buffer the M/G/X tiles;
// long ones (wide ranks) trade that for a deeper operand ring.
template <int OPS, int EPI>
constexpr size_t upd_smem() { return OPS * (size_t)kPStage + EPI * (size_t)kEBuf + 1024 + 256; }

constexpr int kUpdEpiWarps = 8;
constexpr int kUpdThreads = (kUpdEpiWarps + 2) * 32;

template <int OPS, int EPI>
__global__ void __launch_bounds__(kUpdThreads, 1) dion_update_persist_kernel(
    const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmR,
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmM,
    const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmX, UpdPArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* ops = smem;                              // [OPS][kPStage]
    uint8_t* epi = smem + OPS * kPStage;              // [EPI][kEBuf]
    uint64_t* ofull = (uint64_t*)(epi + EPI * kEBuf);
    uint64_t* oempty = ofull + OPS;
    uint64_t* efull = oempty + OPS;
    uint64_t* eempty = efull + EPI;
    uint64_t* afull = eempty + EPI;
    uint64_t* aempty = afull + 2;
    uint32_t* tmem_slot = (uint32_t*)(aempty + 2);
    int* abort_flag = (int*)(tmem_slot + 1);
    volatile int* abrt = abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float one_minus_mu, decay, scale;
    a.hp.get(one_minus_mu, decay, scale);
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0 && !a.hp.finite())
        atomicOr(a.status, kStatusNonFinite);
    const int per_mat = a.tiles_m * a.tiles_n, tiles = a.batch * per_mat;

    if (threadIdx.x == 0) {
        for (int s = 0; s < OPS; ++s) {
            tc::mbar_init(&ofull[s], 1);
            tc::mbar_init(&oempty[s], 1);
        }
        for (int s = 0; s < EPI; ++s) {
            tc::mbar_init(&efull[s], 1);
            tc::mbar_init(&eempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&afull[s], 1);
            tc::mbar_init(&aempty[s], kUpdEpiWarps);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == kUpdEpiWarps + 1) {
        tc::tmem_alloc(tmem_slot, 256);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kUpdEpiWarps) {
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int it = 0;
            for (int t = blockIdx.x; t < tiles && !*abrt; t += gridDim.x, ++it) {
                const int b = t / per_mat, rem = t % per_mat;
                const int m0 = (a.m_fast ? rem % a.tiles_m : rem / a.tiles_n) * kBM;
                const int n0 = (a.m_fast ? rem / a.tiles_m : rem % a.tiles_n) * kUBN;
                const int eb = it % EPI;
                if (!tc::mbar_wait(&eempty[eb], ((it / EPI) & 1) ^ 1, abrt, a.status)) break;
                uint8_t* e = epi + eb * kEBuf;
                tc::mbar_arrive_expect_tx(&efull[eb], kEBuf);
                tc::tma_load_3d(e, &tmM, &efull[eb], n0, m0, b);
                tc::tma_load_3d(e + 16384, &tmM, &efull[eb], n0 + 32, m0, b);
                tc::tma_load_3d(e + kEM, &tmG, &efull[eb], n0, m0, b);
                tc::tma_load_3d(e + kEM + kEG, &tmX, &efull[eb], n0, m0, b);
                for (int kc = 0; kc < a.kchunks; ++kc) {
                    if (!tc::mbar_wait(&oempty[stage], ph ^ 1, abrt, a.status)) break;
                    uint8_t* o = ops + stage * kPStage;
                    tc::mbar_arrive_expect_tx(&ofull[stage], kPStage);
                    tc::tma_load_3d(o, &tmP, &ofull[stage], kc * kBK, m0, b);
                    tc::tma_load_3d(o + kUA, &tmR, &ofull[stage], kc * kBK, n0, b);
                    tc::tma_load_3d(o + kUA + kUB, &tmQ, &ofull[stage], kc * kBK, n0, b);
                    if (++stage == OPS) { stage = 0; ph ^= 1; }
                }
            }
        }
    } else if (warp == kUpdEpiWarps + 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::make_idesc(kBM, kUBN, 1, false, false);
            int stage = 0;
            uint32_t ph = 0;
            int it = 0;
            for (int t = blockIdx.x; t < tiles && !*abrt; t += gridDim.x, ++it) {
                const int ab = it & 1;
                if (!tc::mbar_wait(&aempty[ab], ((it >> 1) & 1) ^ 1, abrt, a.status)) break;
                tc::tc_fence_after();
                const uint32_t d = tmem + ab * 128;
                bool ok = true;
                for (int kc = 0; kc < a.kchunks; ++kc) {
                    if (!tc::mbar_wait(&ofull[stage], ph, abrt, a.status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(ops + stage * kPStage), r0 = a0 + kUA, q0 = r0 + kUB;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t ad = tc::make_sdesc(a0 + k * 32, 16, 1024);
                        tc::mma_bf16(d, ad, tc::make_sdesc(r0 + k * 32, 16, 1024), idesc, (kc | k) != 0);
                        tc::mma_bf16(d + kUBN, ad, tc::make_sdesc(q0 + k * 32, 16, 1024), idesc, (kc | k) != 0);
                    }
                    tc::mma_commit(&oempty[stage]);
                    if (++stage == OPS) { stage = 0; ph ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit(&afull[ab]);
            }
        }
    } else {
        const int quarter = warp & 3, h = warp >> 2;  // TMEM lane quarter, 32-column half
        const int row = quarter * 32 + lane;          // tile row == TMEM lane
        int it = 0;
        for (int t = blockIdx.x; t < tiles && !*abrt; t += gridDim.x, ++it) {
            const int b = t / per_mat, rem = t % per_mat;
            const int m0 = (a.m_fast ? rem % a.tiles_m : rem / a.tiles_n) * kBM;
            const int n0 = (a.m_fast ? rem / a.tiles_m : rem % a.tiles_n) * kUBN;
            const int ab = it & 1, eb = it % EPI;
            const uint32_t aph = (it >> 1) & 1, eph = (it / EPI) & 1;
            const bool ok = tc::mbar_wait(&afull[ab], aph, abrt, a.status) &&
                            tc::mbar_wait(&efull[eb], eph, abrt, a.status);
            tc::tc_fence_after();
            uint8_t* e = epi + eb * kEBuf;
            {
                uint32_t pr[32], pq[32];
                tc::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ab * 128 + h * 32), pr);
                tc::tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ab * 128 + kUBN + h * 32), pq);
                tc::tmem_ld_wait();
                if (ok) {
                uint8_t* eM = e + h * 16384;
#pragma unroll
                for (int c = 0; c < 8; ++c) {        // M: 8 chunks of 4 floats
                    float4* pm = reinterpret_cast<float4*>(eM + tc::sw128_offset(row, c));
                    const uint32_t gchunk = h * 4 + (c >> 1);
                    const bf16* gh = reinterpret_cast<const bf16*>(e + kEM + tc::sw128_offset(row, gchunk)) + (c & 1) * 4;
                    float4 mv = *pm;
                    mv.x = mv.x + __bfloat162float(gh[0]) - one_minus_mu * __uint_as_float(pr[4 * c + 0]);
                    mv.y = mv.y + __bfloat162float(gh[1]) - one_minus_mu * __uint_as_float(pr[4 * c + 1]);
                    mv.z = mv.z + __bfloat162float(gh[2]) - one_minus_mu * __uint_as_float(pr[4 * c + 2]);
                    mv.w = mv.w + __bfloat162float(gh[3]) - one_minus_mu * __uint_as_float(pr[4 * c + 3]);
                    *pm = mv;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {        // X: 4 chunks of 8 bf16
                    uint4* px = reinterpret_cast<uint4*>(e + kEM + kEG + tc::sw128_offset(row, h * 4 + c));
                    uint4 xv = *px;
                    const bf16* xh = reinterpret_cast<const bf16*>(&xv);
                    float o[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        o[q] = decay * __bfloat162float(xh[q]) - scale * __uint_as_float(pq[8 * c + q]);
                    *px = pack8(o);
                }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&aempty[ab]);
            tc::fence_proxy_async_smem();
            tc::named_bar_sync(1, kUpdEpiWarps * 32);
            if (threadIdx.x == 0) {
                if (ok) {
                    tc::tma_store_3d(&tmM, e, n0, m0, b);
                    tc::tma_store_3d(&tmM, e + 16384, n0 + 32, m0, b);
                    tc::tma_store_3d(&tmX, e + kEM + kEG, n0, m0, b);
                    tc::tma_store_commit();
                    tc::tma_store_wait_read();
                }
                tc::mbar_arrive(&eempty[eb]);
            }
        }
        if (threadIdx.x == 0) tc::tma_store_wait_all();
    }
    __syncthreads();
    if (warp == kUpdEpiWarps + 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 256);
    }
}

// ------------------------------- wide-rank M update (256 < rp <= 512)
// M <- M + G - (1 - mu) P R^T over 128 x 128 tiles of M with K = rp, as a
// persistent kernel.  The P and R chunks stream through four 32 KB operand
// stages.  M and G move by TMA in 32-column blocks through a ring of four
// 24 KB slots that a warp of its own keeps loaded, so about three blocks of
// M and G (72 KB) are in flight per SM without holding registers; each
// block's result overwrites its M in shared memory and is stored by TMA.
//   warp 0: operand producer   warp 1: MMA issuer   warp 2: M/G block loader
//   warps 3..10: epilogue (warp w: TMEM lane quarter w % 4, 16-column half
//   (w - 3) / 4 of each block)
constexpr int kMwBN = 128, kMwOps = 4, kMwSlots = 4, kMwEpiWarps = 8;
constexpr int kMwEpiWarp0 = 3;
constexpr int kMwThreads = (kMwEpiWarp0 + kMwEpiWarps) * 32;
constexpr int kMwBlocks = kMwBN / 32;                              // 32-column blocks per tile
constexpr uint32_t kMwA = kBM * kBK * 2;                           // 16 KB P chunk
constexpr uint32_t kMwStage = kMwA + kMwBN * kBK * 2;              // + 16 KB R chunk
constexpr uint32_t kMwM = kBM * 32 * 4, kMwG = kBM * 32 * 2;       // 16 KB of M, 8 KB of G per block
constexpr uint32_t kMwSlot = kMwM + kMwG;
constexpr size_t kMwSmem = (size_t)kMwOps * kMwStage + (size_t)kMwSlots * kMwSlot + 1024 + 256;
static_assert(kMwSmem <= 232448, "shared memory per CTA");
static_assert(kMwSlot % 1024 == 0 && kMwM % 1024 == 0, "swizzled boxes need 1024-byte aligned slots");

struct MwArgs {
    int m, n, batch, kchunks, tiles_m, tiles_n;
    StepHyper hp;
    int* status;
    int m_fast;   // row tiles fastest (see UpdPArgs)
};

// byte offset of 16-byte chunk `chunk` (0..3) of row `row` in a box of
// 64-byte rows stored with the 64-byte swizzle
__device__ __forceinline__ uint32_t sw64_offset(uint32_t row, uint32_t chunk)
{
    return row * 64u + ((chunk ^ ((row >> 1) & 3u)) << 4);
}

__global__ void __launch_bounds__(kMwThreads, 1) dion_update_mwide_kernel(
    const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmR,
    const __grid_constant__ CUtensorMap tmM, const __grid_constant__ CUtensorMap tmG, MwArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* ops = smem;                                  // [kMwOps][kMwStage]
    uint8_t* slots = smem + kMwOps * kMwStage;            // [kMwSlots][kMwSlot]
    uint64_t* ofull = (uint64_t*)(slots + kMwSlots * kMwSlot);
    uint64_t* oempty = ofull + kMwOps;
    uint64_t* efull = oempty + kMwOps;
    uint64_t* eempty = efull + kMwSlots;
    uint64_t* afull = eempty + kMwSlots;
    uint64_t* aempty = afull + 2;
    uint32_t* tmem_slot = (uint32_t*)(aempty + 2);
    int* abort_flag = (int*)(tmem_slot + 1);
    volatile int* abrt = abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float one_minus_mu, decay, scale;
    a.hp.get(one_minus_mu, decay, scale);
    if (blockIdx.x == 0 && threadIdx.x == 0 && !a.hp.finite()) atomicOr(a.status, kStatusNonFinite);
    const int per_mat = a.tiles_m * a.tiles_n, tiles = a.batch * per_mat;
    auto tile_of = [&](int t, int& b, int& m0, int& n0) {
        b = t / per_mat;
        const int rem = t % per_mat;
        m0 = (a.m_fast ? rem % a.tiles_m : rem / a.tiles_n) * kBM;
        n0 = (a.m_fast ? rem / a.tiles_m : rem % a.tiles_n) * kMwBN;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMwOps; ++s) {
            tc::mbar_init(&ofull[s], 1);
            tc::mbar_init(&oempty[s], 1);
        }
        for (int s = 0; s < kMwSlots; ++s) {
            tc::mbar_init(&efull[s], 1);
            tc::mbar_init(&eempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            tc::mbar_init(&afull[s], 1);
            tc::mbar_init(&aempty[s], kMwEpiWarps);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 2 * kMwBN);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok && !*abrt; t += gridDim.x) {
                int b, m0, n0;
                tile_of(t, b, m0, n0);
                for (int kc = 0; kc < a.kchunks; ++kc) {
                    if (!tc::mbar_wait(&oempty[stage], ph ^ 1, abrt, a.status)) { ok = false; break; }
                    uint8_t* o = ops + stage * kMwStage;
                    tc::mbar_arrive_expect_tx(&ofull[stage], kMwStage);
                    tc::tma_load_3d(o, &tmP, &ofull[stage], kc * kBK, m0, b);
                    tc::tma_load_3d(o + kMwA, &tmR, &ofull[stage], kc * kBK, n0, b);
                    if (++stage == kMwOps) { stage = 0; ph ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::make_idesc(kBM, kMwBN, 1, false, false);
            int stage = 0, it = 0;
            uint32_t ph = 0;
            for (int t = blockIdx.x; t < tiles && !*abrt; t += gridDim.x, ++it) {
                const int ab = it & 1;
                if (!tc::mbar_wait(&aempty[ab], ((it >> 1) & 1) ^ 1, abrt, a.status)) break;
                tc::tc_fence_after();
                const uint32_t d = tmem + ab * kMwBN;
                bool ok = true;
                for (int kc = 0; kc < a.kchunks; ++kc) {
                    if (!tc::mbar_wait(&ofull[stage], ph, abrt, a.status)) { ok = false; break; }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(ops + stage * kMwStage), r0 = a0 + kMwA;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc::mma_bf16(d, tc::make_sdesc(a0 + k * 32, 16, 1024), tc::make_sdesc(r0 + k * 32, 16, 1024),
                                     idesc, (kc | k) != 0);
                    tc::mma_commit(&oempty[stage]);
                    if (++stage == kMwOps) { stage = 0; ph ^= 1; }
                }
                if (!ok) break;
                tc::mma_commit(&afull[ab]);
            }
        }
    } else if (warp == 2) {
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok && !*abrt; t += gridDim.x) {
                int b, m0, n0;
                tile_of(t, b, m0, n0);
                for (int blk = 0; blk < kMwBlocks; ++blk, ++g) {
                    const int s = g % kMwSlots;
                    if (!tc::mbar_wait(&eempty[s], ((g / kMwSlots) & 1) ^ 1, abrt, a.status)) { ok = false; break; }
                    uint8_t* e = slots + s * kMwSlot;
                    tc::mbar_arrive_expect_tx(&efull[s], kMwSlot);
                    tc::tma_load_3d(e, &tmM, &efull[s], n0 + 32 * blk, m0, b);
                    tc::tma_load_3d(e + kMwM, &tmG, &efull[s], n0 + 32 * blk, m0, b);
                }
            }
        }
    } else {
        // The trip counts here do not depend on the abort flag (every wait
        // returns at once after an abort), so all epilogue warps pass the
        // same named barriers.
        const int quarter = warp & 3, h = (warp - kMwEpiWarp0) >> 2;
        const uint32_t row = quarter * 32 + lane;     // tile row == TMEM lane
        const bool leader = threadIdx.x == kMwEpiWarp0 * 32;
        int it = 0, g = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            int b, m0, n0;
            tile_of(t, b, m0, n0);
            const int ab = it & 1;
            bool ok = tc::mbar_wait(&afull[ab], (it >> 1) & 1, abrt, a.status);
            tc::tc_fence_after();
            for (int blk = 0; blk < kMwBlocks; ++blk, ++g) {
                const int s = g % kMwSlots;
                ok = tc::mbar_wait(&efull[s], (g / kMwSlots) & 1, abrt, a.status) && ok;
                uint8_t* e = slots + s * kMwSlot;
                uint32_t pr[16];
                tc::tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(ab * kMwBN + blk * 32 + h * 16), pr);
                tc::tmem_ld_wait();
                if (ok) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {   // columns h * 16 + 4c .. + 3 of the block
                        float4* pm = reinterpret_cast<float4*>(e + tc::sw128_offset(row, h * 4 + c));
                        const bf16* gh =
                            reinterpret_cast<const bf16*>(e + kMwM + sw64_offset(row, h * 2 + (c >> 1))) + (c & 1) * 4;
                        float4 mv = *pm;
                        mv.x = mv.x + __bfloat162float(gh[0]) - one_minus_mu * __uint_as_float(pr[4 * c + 0]);
                        mv.y = mv.y + __bfloat162float(gh[1]) - one_minus_mu * __uint_as_float(pr[4 * c + 1]);
                        mv.z = mv.z + __bfloat162float(gh[2]) - one_minus_mu * __uint_as_float(pr[4 * c + 2]);
                        mv.w = mv.w + __bfloat162float(gh[3]) - one_minus_mu * __uint_as_float(pr[4 * c + 3]);
                        *pm = mv;
                    }
                }
                tc::fence_proxy_async_smem();
                tc::named_bar_sync(1, kMwEpiWarps * 32);
                if (leader) {
                    if (ok) {
                        tc::tma_store_3d(&tmM, e, n0 + 32 * blk, m0, b);
                        tc::tma_store_commit();
                        tc::tma_store_wait_read();
                    }
                    tc::mbar_arrive(&eempty[s]);
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&aempty[ab]);
        }
        if (leader) tc::tma_store_wait_all();
    }
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 2 * kMwBN);
    }
}

// ------------------------------------------------------------ small kernels

// Qt[b][j][k] = bf16(Q[b][k][j]) for j < r; zero rows r <= j < rp.
__global__ void __launch_bounds__(256) dion_prep_qt_kernel(int n, int r, int rp, long long ldqt, const float* Q,
                                                           bf16* Qt, int* counter)
{
    __shared__ float tile[32][33];
    const int b = blockIdx.z, k0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && threadIdx.y == 0) counter[b] = 0;   // for dion_rsum
    for (int kk = threadIdx.y; kk < 32; kk += 8) {
        const int k = k0 + kk, j = j0 + threadIdx.x;
        tile[kk][threadIdx.x] = (k < n && j < r) ? Q[((long long)b * n + k) * r + j] : 0.f;
    }
    __syncthreads();
    for (int jj = threadIdx.y; jj < 32; jj += 8) {
        const int j = j0 + jj, k = k0 + threadIdx.x;
        if (j < rp && k < n) Qt[((long long)b * rp + j) * ldqt + k] = __float2bfloat16_rn(tile[threadIdx.x][jj]);
    }
}

// ------------------------------------------------- wide ranks (rp > 256)
// B = M + G as bf16 once, row-major (B16, pitch pb), for the two TMA GEMMs
// that replace the fused passes when the rank spans several 256-column chunks
// (the fused passes would re-read M and G once per chunk): B Q reads it
// K-major, B^T P MN-major.  One thread per 16 consecutive elements of a row.
template <bool VEC>
__global__ void __launch_bounds__(256) dion_formb_kernel(int m, int n, long long pb, const float* M, const bf16* G,
                                                         bf16* B16)
{
    const int b = blockIdx.z, c0 = blockIdx.x * 64, i0 = blockIdx.y * 64;
    const size_t base = (size_t)b * m * n;
    const int ri = threadIdx.x >> 2, cg = (threadIdx.x & 3) * 16, i = i0 + ri, c = c0 + cg;
    if (i >= m || c >= n) return;
    float v[16];
    if (VEC && c + 16 <= n) {
        const float* mr = M + base + (size_t)i * n + c;
        const bf16* gr = G + base + (size_t)i * n + c;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(mr + 4 * q));
            v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint4 g = __ldg(reinterpret_cast<const uint4*>(gr + 8 * q));
            const bf16* h = reinterpret_cast<const bf16*>(&g);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[8 * q + e] += __bfloat162float(h[e]);
        }
        bf16* o = B16 + (size_t)b * m * pb + (size_t)i * pb + c;
        *reinterpret_cast<uint4*>(o) = make_uint4(tc::pack_bf16x2(v[0], v[1]), tc::pack_bf16x2(v[2], v[3]),
                                                  tc::pack_bf16x2(v[4], v[5]), tc::pack_bf16x2(v[6], v[7]));
        *reinterpret_cast<uint4*>(o + 8) = make_uint4(tc::pack_bf16x2(v[8], v[9]), tc::pack_bf16x2(v[10], v[11]),
                                                      tc::pack_bf16x2(v[12], v[13]), tc::pack_bf16x2(v[14], v[15]));
    } else {
        bf16* o = B16 + (size_t)b * m * pb + (size_t)i * pb;
        for (int e = 0; e < 16 && c + e < n; ++e) {
            const size_t x = base + (size_t)i * n + c + e;
            o[c + e] = __float2bfloat16_rn(M[x] + __bfloat162float(G[x]));
        }
    }
}


// Q16 = bf16(Q) (n x rp, row-major, padding columns zero): the MN-major
// operand of B Q (rp <= 256).  Four columns per thread.  Also zeroes the
// column-norm arrival counters of dion_rsum for this step.
__global__ void __launch_bounds__(256) dion_prep_q16_kernel(int n, int r, int rp, const float* __restrict__ Q,
                                                            bf16* __restrict__ Q16, int* counter)
{
    const int b = blockIdx.y, upr = rp >> 2, total = n * upr;
    if (blockIdx.x == 0 && threadIdx.x == 0) counter[b] = 0;
    const float* Qb = Q + (size_t)b * n * r;
    bf16* Ob = Q16 + (size_t)b * n * rp;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        const int j = e / upr, c = (e - j * upr) * 4;
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = (c + t < r) ? Qb[(size_t)j * r + c + t] : 0.f;
        *reinterpret_cast<uint2*>(Ob + (size_t)j * rp + c) =
            make_uint2(tc::pack_bf16x2(v[0], v[1]), tc::pack_bf16x2(v[2], v[3]));
    }
}

constexpr int kRChunk = 32;

// R = sum of the split partials (fp32, pitch rp), R16 = bf16(R) (columns r..rp-1
// zero), and per-chunk column sums of squares normpart[b][chunk][c] over rows
// chunk*kRChunk ..: every sum in a fixed order, so results are reproducible.
// The CTA that finishes last for matrix b (a per-matrix arrival counter,
// zeroed by dion_prep_qt_kernel earlier in the step) reduces the chunks in
// order into inv[b][c] = 1 / max(||R_c||, floor) (0 for padding columns) and
// resets the counter.
// kCopy = false: the B^T P GEMM already wrote R and R16; part is R itself
// (one partial) and only the column norms are formed.
template <bool kCopy>
__global__ void __launch_bounds__(256) dion_rsum_kernel(int n, int r, int rp, int splits, int batch,
                                                        const float* __restrict__ part, float* __restrict__ R,
                                                        bf16* __restrict__ R16, float* __restrict__ normpart,
                                                        int* counter, float* inv, float floor_nrm, int* status)
{
    __shared__ int s_last;
    __shared__ float4 s_ss[4][64];
    const int b = blockIdx.y, chunk = blockIdx.x, nchunks = gridDim.x;
    const int j0 = chunk * kRChunk;
    const long long pstride = (long long)batch * n * rp;
    // thread = 4 columns (cg) x rows j0 + rl, j0 + rl + 4, ... (8 rows): float4
    // accesses; 256 columns per pass over the rp columns
    const int cg = threadIdx.x & 63, rl = threadIdx.x >> 6;
    for (int cb = 0; cb < rp; cb += 256) {
    const int c = cb + cg * 4;
    float4 ss = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < rp) {
        float4 v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int j = j0 + rl + 4 * t;
            v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < n) {
                const long long o = ((long long)b * n + j) * rp + c;
                v[t] = *reinterpret_cast<const float4*>(part + o);
                for (int q = 1; q < splits; ++q) {
                    const float4 u = *reinterpret_cast<const float4*>(part + o + q * pstride);
                    v[t].x += u.x; v[t].y += u.y; v[t].z += u.z; v[t].w += u.w;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int j = j0 + rl + 4 * t;
            if (j < n) {
                float4 x = v[t];
                if (c >= r) x.x = 0.f;
                if (c + 1 >= r) x.y = 0.f;
                if (c + 2 >= r) x.z = 0.f;
                if (c + 3 >= r) x.w = 0.f;
                const long long o = ((long long)b * n + j) * rp + c;
                if (kCopy) {
                    *reinterpret_cast<float4*>(R + o) = x;
                    *reinterpret_cast<uint2*>(R16 + o) =
                        make_uint2(tc::pack_bf16x2(x.x, x.y), tc::pack_bf16x2(x.z, x.w));
                }
                ss.x = fmaf(x.x, x.x, ss.x); ss.y = fmaf(x.y, x.y, ss.y);
                ss.z = fmaf(x.z, x.z, ss.z); ss.w = fmaf(x.w, x.w, ss.w);
            }
        }
    }
    s_ss[rl][cg] = ss;
    __syncthreads();
    if (rl == 0 && c < rp) {   // the four row lanes, in a fixed order
        const float4 a0 = s_ss[0][cg], a1 = s_ss[1][cg], a2 = s_ss[2][cg], a3 = s_ss[3][cg];
        *reinterpret_cast<float4*>(normpart + ((long long)b * nchunks + chunk) * rp + c) =
            make_float4((a0.x + a1.x) + (a2.x + a3.x), (a0.y + a1.y) + (a2.y + a3.y), (a0.z + a1.z) + (a2.z + a3.z),
                        (a0.w + a1.w) + (a2.w + a3.w));
    }
    __syncthreads();
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&counter[b], 1) == nchunks - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int c = threadIdx.x; c < rp; c += blockDim.x) {
        // eight interleaved partial sums (loads in flight), combined in a fixed order
        const float* np_ = normpart + (long long)b * nchunks * rp + c;
        float t8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int k = 0;
        for (; k + 8 <= nchunks; k += 8) {
#pragma unroll
            for (int q = 0; q < 8; ++q) t8[q] += __ldcg(np_ + (long long)(k + q) * rp);
        }
        for (; k < nchunks; ++k) t8[k & 7] += __ldcg(np_ + (long long)k * rp);
        const float t = ((t8[0] + t8[1]) + (t8[2] + t8[3])) + ((t8[4] + t8[5]) + (t8[6] + t8[7]));
        float v = 0.f;
        if (c < r) {
            v = 1.f / fmaxf(sqrtf(t), floor_nrm);
            if (!isfinite(t)) atomicOr(status, kStatusNonFinite);
        }
        inv[(long long)b * rp + c] = v;
    }
    if (threadIdx.x == 0) counter[b] = 0;
}

// Q = R * inv (the caller's n x r float32 state) and Q16 = bf16(Q) (n x rp
// operand), four columns per thread.
__global__ void __launch_bounds__(256) dion_qemit_kernel(int n, int r, int rp, int rows,
                                                         const float* __restrict__ R, const float* __restrict__ inv,
                                                         float* __restrict__ Q, bf16* __restrict__ Q16, bool qvec)
{
    const int upr = rp >> 2;
    const int total = rows * upr;                     // rows = batch * n
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        const int row = e / upr, c = (e - row * upr) * 4, b = row / n;
        const float4 x = *reinterpret_cast<const float4*>(R + (size_t)row * rp + c);
        const float4 s = *reinterpret_cast<const float4*>(inv + (size_t)b * rp + c);
        const float q[4] = {x.x * s.x, x.y * s.y, x.z * s.z, x.w * s.w};
        *reinterpret_cast<uint2*>(Q16 + (size_t)row * rp + c) =
            make_uint2(tc::pack_bf16x2(q[0], q[1]), tc::pack_bf16x2(q[2], q[3]));
        float* qo = Q + (size_t)row * r + c;
        if (qvec) {   // r % 4 == 0 and Q 16-byte aligned: whole quads below r
            if (c < r) *reinterpret_cast<float4*>(qo) = make_float4(q[0], q[1], q[2], q[3]);
        } else {
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (c + t < r) qo[t] = q[t];
        }
    }
}

}  // namespace

static unsigned grid_for(long long work, int per = 256 * 4)
{
    long long g = cdiv(work, per);
    if (g < 1) g = 1;
    if (g > 65535) g = 65535;
    return (unsigned)g;
}

template <bool MN_A>
static cudaError_t launch_pass(const char* name, bool vec, const CUtensorMap& tm, const CUtensorMap& tms,
                               const PassArgs& pa, cudaStream_t st)
{
    const int out_rows = MN_A ? pa.n : pa.m;
    const long long units = cdiv(out_rows, kBM) * (long long)pa.splits * pa.batch;
    const dim3 grid((unsigned)std::min<long long>(units, num_sms()));
    static std::atomic<unsigned long long> attr[2] = {{0}, {0}};
    auto k = vec ? dion_pass_kernel<MN_A, true> : dion_pass_kernel<MN_A, false>;
    cudaError_t e = smem_attr_once((const void*)k, (int)kPassSmem, attr[vec]);
    if (e != cudaSuccess) return e;
    return launch(name, k, grid, dim3(kPassWarps * 32), kPassSmem, st, tm, tms, pa);
}

dion_status dion_step_tc(int batch, int m, int n, int r, void* Xv, const void* Gv, float* M, float* Q, float mu,
                         float lr, float wd, const float* hyper, char* ws, const DionLayout& L, cudaStream_t st)
{
    const StepHyper hp{mu, lr, wd, sqrtf((float)m / (float)n), hyper};
    bf16* X = (bf16*)Xv;
    const bf16* G = (const bf16*)Gv;
    const int rp = L.rp;
    int* status = (int*)(ws + L.status);
    float* part = (float*)(ws + L.Ppart);
    float* P0 = (float*)(ws + L.P0);
    float* P1 = (float*)(ws + L.P1);
    float* R = (float*)(ws + L.R);
    float* inv = (float*)(ws + L.inv);
    bf16* Qt16 = (bf16*)(ws + L.Qt16);
    bf16* P16 = (bf16*)(ws + L.P16);
    bf16* R16 = (bf16*)(ws + L.R16);
    bf16* Q16 = (bf16*)(ws + L.Q16);
    float* normp = (float*)(ws + L.normp);
    const long long np = (long long)align_up((size_t)n, 8);
    const bool vec = (n % 8) == 0;

    DION_TRY(cudaMemsetAsync(status, 0, sizeof(int), st));
    // 1. Qt = bf16(Q^T)
    int* rcount = (int*)(ws + L.rcount);
    const float floor_nrm = 1e-12f * sqrtf((float)n);
    if (L.wide) {   // 1. Qt = bf16(Q^T), the K-major operand of the B Q GEMM
        DION_TRY(launch("dion_prep_qt", dion_prep_qt_kernel, dim3((unsigned)cdiv(n, 32), (unsigned)cdiv(rp, 32), batch),
                        dim3(32, 8), 0, st, n, r, rp, np, (const float*)Q, Qt16, rcount));
    } else {        // 1. Q16 = bf16(Q), the MN-major operand of the fused pass
        DION_TRY(launch("dion_prep_qt", dion_prep_q16_kernel,
                        dim3((unsigned)std::min<long long>(cdiv((long long)n * (rp / 4), 256), 1024), batch), dim3(256),
                        0, st, n, r, rp, (const float*)Q, Q16, rcount));
    }
    if (L.wide) {
        // 2'. B = M + G once in bf16 (and B^T); P = B Q as a TMA GEMM into part (one split)
        bf16* B16 = (bf16*)(ws + L.B16);
        // B in bf16, row-major only: B^T P below reads it MN-major
        auto fk = vec ? dion_formb_kernel<true> : dion_formb_kernel<false>;
        DION_TRY(launch("dion_formb", fk, dim3((unsigned)cdiv(n, 64), (unsigned)cdiv(m, 64), batch), dim3(256), 0, st, m,
                        n, np, (const float*)M, G, B16));
        CUtensorMap tA, tB;
        if (!make_tmap_3d(&tA, B16, TmapType::BF16, n, m, batch, np * 2, (long long)m * np * 2, 64, kBM) ||
            !make_tmap_3d(&tB, Qt16, TmapType::BF16, n, rp, batch, np * 2, rp * np * 2, 64, 256))
            return DION_ERR_CUDA;
        TcGemmEpi e{};
        e.M = m; e.N = rp; e.tiles_m = (int)cdiv(m, kBM); e.tiles_n = (int)cdiv(rp, 256); e.batch = batch;
        e.Cf = part; e.ldc = rp; e.sc = (long long)m * rp; e.alpha = 0.f; e.beta = 1.f; e.status = status;
        e.nseg = 1; e.zmul = 1;
        DION_TRY(tc_gemm<256>("dion_bq_tc", tA, tB, n, e, st));
        DION_TRY(qr_cholesky2_tc(batch, m, r, rp, part, 1, P0, P1, P16, ws, L, status, st, n, M, G, Q));
        // 6'. R = B^T P: A = B^T read MN-major from the row-major bf16 B (64 x 64
        // boxes), B operand = P16 read MN-major; no transposed copies
        CUtensorMap tA2, tB2;
        if (!make_tmap_3d(&tA2, B16, TmapType::BF16, n, m, batch, np * 2, (long long)m * np * 2, 64, 64) ||
            !make_tmap_3d(&tB2, P16, TmapType::BF16, rp, m, batch, (long long)rp * 2, (long long)m * rp * 2, 64, 64))
            return DION_ERR_CUDA;
        TcGemmEpi e2 = e;
        e2.M = n; e2.tiles_m = (int)cdiv(n, kBM); e2.sc = (long long)n * rp;
        e2.Cf = R; e2.C = R16;   // R (float32) and R16 straight from the epilogue (P16's columns past r are zero)
        DION_TRY((tc_gemm<256, true>("dion_btp_tc", tA2, tB2, m, e2, st)));
        const int nchunks = (int)cdiv(n, kRChunk);
        DION_TRY(launch("dion_rsum", dion_rsum_kernel<false>, dim3((unsigned)nchunks, batch), dim3(256), 0, st, n, r,
                        rp, 1, batch, (const float*)R, R, R16, normp, rcount, inv, floor_nrm, status));
    } else {
    // 2. P partials = B Q (with n % 8 == 0 the pass also stores B in bf16)
    CUtensorMap tmQt;
    if (!make_tmap_3d(&tmQt, Q16, TmapType::BF16, rp, n, batch, (long long)rp * 2, (long long)n * rp * 2, 64, 64))
        return DION_ERR_CUDA;
    bf16* B16 = L.b16_narrow ? (bf16*)(ws + L.B16) : nullptr;
    CUtensorMap tmS = tmQt;   // where the B Q pass stores bf16 B (unused without B16)
    if (B16 && !make_tmap_3d(&tmS, B16, TmapType::BF16, n, m, batch, (long long)n * 2, (long long)m * n * 2, 64, kBM))
        return DION_ERR_CUDA;
    {
        const int kchunks = (int)cdiv(n, kBK);
        const int kcps = (int)cdiv(kchunks, L.ksplit);
        const int splits = (int)cdiv(kchunks, kcps);
        // one split: the epilogue writes the terms of P (and, for the blocked
        // factorization, P as float32) for the first CholeskyQR pass directly
        const bool terms = splits == 1;
        PassArgs pa{m, n, rp, batch, splits, kcps, kchunks, M, G, part, status, B16 != nullptr,
                    terms ? (bf16*)(ws + L.P3) : nullptr, (terms && L.nbc > 0) ? P1 : nullptr};
        DION_TRY(launch_pass<false>("dion_bq_tc", vec, tmQt, tmS, pa, st));
        // 3-5. CholeskyQR2; its first pass reads the split partials of P directly (or the
        // terms above), its last product writes P (float32, P0) and P16 = bf16(P)
        DION_TRY(qr_cholesky2_tc(batch, m, r, rp, part, splits, P0, P1, P16, ws, L, status, st, n, M, G, Q, terms));
    }
    // 6. R partials = B^T P
    const int nchunks = (int)cdiv(n, kRChunk);
    if (B16) {
        // as a TMA GEMM on the stored bf16 B: A = B^T read MN-major from the
        // row-major B (64 x 64 boxes), B operand = P16 read MN-major; one split
        CUtensorMap tA, tB;
        const int bn = rp <= 64 ? 64 : (rp <= 128 ? 128 : (rp <= 192 ? 192 : 256));
        if (!make_tmap_3d(&tA, B16, TmapType::BF16, n, m, batch, (long long)n * 2, (long long)m * n * 2, 64, 64) ||
            !make_tmap_3d(&tB, P16, TmapType::BF16, rp, m, batch, (long long)rp * 2, (long long)m * rp * 2, 64, 64))
            return DION_ERR_CUDA;
        TcGemmEpi e{};
        e.M = n; e.N = rp; e.tiles_m = (int)cdiv(n, kBM); e.tiles_n = (int)cdiv(rp, bn); e.batch = batch;
        e.Cf = R; e.C = R16; e.ldc = rp; e.sc = (long long)n * rp; e.alpha = 0.f; e.beta = 1.f; e.status = status;
        e.nseg = 1; e.zmul = 1;
        cudaError_t ce;
        if (bn == 64) ce = tc_gemm<64, true>("dion_btp_tc", tA, tB, m, e, st);
        else if (bn == 128) ce = tc_gemm<128, true>("dion_btp_tc", tA, tB, m, e, st);
        else if (bn == 192) ce = tc_gemm<192, true>("dion_btp_tc", tA, tB, m, e, st);
        else ce = tc_gemm<256, true>("dion_btp_tc", tA, tB, m, e, st);
        DION_TRY(ce);
        // 7. column norms of R (the GEMM wrote R and R16; P16's columns past r are zero)
        DION_TRY(launch("dion_rsum", dion_rsum_kernel<false>, dim3((unsigned)nchunks, batch), dim3(256), 0, st, n, r,
                        rp, 1, batch, (const float*)R, R, R16, normp, rcount, inv, floor_nrm, status));
    } else {
        CUtensorMap tmP64;
        if (!make_tmap_3d(&tmP64, P16, TmapType::BF16, rp, m, batch, (long long)rp * 2, (long long)m * rp * 2, 64, 64))
            return DION_ERR_CUDA;
        const int kchunks = (int)cdiv(m, kBK);
        const int kcps = (int)cdiv(kchunks, L.ksplit_r);
        const int splits = (int)cdiv(kchunks, kcps);
        PassArgs pa{m, n, rp, batch, splits, kcps, kchunks, M, G, part, status, false, nullptr, nullptr};
        DION_TRY(launch_pass<true>("dion_btp_tc", vec, tmP64, tmP64, pa, st));
        // 7. R = sum of partials, R16, column norms, Q = R / ||R_j||, Q16
        DION_TRY(launch("dion_rsum", dion_rsum_kernel<true>, dim3((unsigned)nchunks, batch), dim3(256), 0, st, n, r,
                        rp, splits, batch, (const float*)part, R, R16, normp, rcount, inv, floor_nrm, status));
    }
    }
    {
        const int rows = batch * n;
        DION_TRY(launch("dion_qemit", dion_qemit_kernel, dim3(grid_for((long long)rows * (rp / 4))), dim3(256), 0, st,
                        n, r, rp, rows, (const float*)R, (const float*)inv, Q, Q16,
                        (r % 4) == 0 && ((uintptr_t)Q & 15u) == 0));
    }
    // 9. M and X updates
    CUtensorMap tmPa, tmR, tmQ;
    if (!make_tmap_3d(&tmPa, P16, TmapType::BF16, rp, m, batch, (long long)rp * 2, (long long)m * rp * 2, 64, kBM) ||
        !make_tmap_3d(&tmR, R16, TmapType::BF16, rp, n, batch, (long long)rp * 2, (long long)n * rp * 2, 64, kUBN) ||
        !make_tmap_3d(&tmQ, Q16, TmapType::BF16, rp, n, batch, (long long)rp * 2, (long long)n * rp * 2, 64, kUBN))
        return DION_ERR_CUDA;
    if (vec && L.wide) {
        // wide ranks: the two products as persistent kernels with the updates
        // in their epilogues (M and X in place):
        //   M <- M + G - (1 - mu) P R^T
        //     rp <= 512: dion_update_mwide_kernel (128 x 128 tiles; M and G move
        //       by TMA through a ring of 32-column blocks)
        //     rp > 512: 128 x 256 TMA GEMM with the coalesced epilogue.  There
        //       the P and R reads from L2 (2 rp (1/128 + 1/BN) bytes per element)
        //       outweigh the 10 bytes of M and G, and the wider tile reads fewer
        //   X <- (1 - lr wd) X - lr sqrt(m/n) P Q^T   128 x 256 TMA GEMM with the
        //     coalesced epilogue, a whole tile's X loaded ahead (bound by its MMAs)
        const long long mn = (long long)m * n;
        CUtensorMap tP, tQb;
        if (!make_tmap_3d(&tP, P16, TmapType::BF16, rp, m, batch, (long long)rp * 2, (long long)m * rp * 2, 64, kBM) ||
            !make_tmap_3d(&tQb, Q16, TmapType::BF16, rp, n, batch, (long long)rp * 2, (long long)n * rp * 2, 64, 256))
            return DION_ERR_CUDA;
        if (rp > 512) {
            CUtensorMap tRb;
            if (!make_tmap_3d(&tRb, R16, TmapType::BF16, rp, n, batch, (long long)rp * 2, (long long)n * rp * 2, 64, 256))
                return DION_ERR_CUDA;
            TcGemmEpi e1{};
            e1.M = m; e1.N = n; e1.tiles_m = (int)cdiv(m, kBM); e1.tiles_n = (int)cdiv(n, 256); e1.batch = batch;
            e1.Cf = M; e1.ldc = n; e1.sc = mn;
            e1.auxf = M; e1.ldauxf = n; e1.sauxf = mn; e1.alpha = 1.f;
            e1.aux2 = G; e1.ldaux2 = n; e1.saux2 = mn; e1.alpha2 = 1.f;
            e1.hp = hp; e1.hp_mode = 1; e1.status = status; e1.nseg = 1; e1.zmul = 1;
            e1.m_fast = e1.tiles_m < e1.tiles_n;
            DION_TRY((tc_gemm<256, false, 8, 1>("dion_update_tc", tP, tRb, rp, e1, st)));
        } else {
            CUtensorMap tR128, tMb, tGb;
            if (!make_tmap_3d(&tR128, R16, TmapType::BF16, rp, n, batch, (long long)rp * 2, (long long)n * rp * 2, 64,
                              kMwBN) ||
                !make_tmap_3d(&tMb, M, TmapType::F32, n, m, batch, (long long)n * 4, mn * 4, 32, kBM) ||
                !make_tmap_3d_sw64(&tGb, G, TmapType::BF16, n, m, batch, (long long)n * 2, mn * 2, 32, kBM))
                return DION_ERR_CUDA;
            const int tm = (int)cdiv(m, kBM), tn = (int)cdiv(n, kMwBN);
            const long long tiles = (long long)tm * tn * batch;
            const int grid = (int)std::min<long long>(tiles, num_sms());
            MwArgs ma{m, n, batch, (int)cdiv(rp, kBK), tm, tn, hp, status, tm < tn ? 1 : 0};
            static std::atomic<unsigned long long> mattr{0};
            DION_TRY(smem_attr_once((const void*)dion_update_mwide_kernel, (int)kMwSmem, mattr));
            DION_TRY(launch("dion_update_tc", dion_update_mwide_kernel, dim3(grid), dim3(kMwThreads), kMwSmem, st,
                            tP, tR128, tMb, tGb, ma));
        }
        TcGemmEpi e2{};
        e2.M = m; e2.N = n; e2.tiles_m = (int)cdiv(m, kBM); e2.tiles_n = (int)cdiv(n, 256); e2.batch = batch;
        e2.C = X; e2.ldc = n; e2.sc = mn;
        e2.aux = X; e2.ldaux = n; e2.saux = mn;
        e2.hp = hp; e2.hp_mode = 2; e2.status = status; e2.nseg = 1; e2.zmul = 1;
        e2.m_fast = e2.tiles_m < e2.tiles_n;
        DION_TRY((tc_gemm<256, false, 8, 2>("dion_update_tc", tP, tQb, rp, e2, st)));
    } else if (vec) {
        // persistent TMA-epilogue pass (needs 16-byte aligned rows of M, G, X)
        CUtensorMap tmM, tmG, tmX;
        const long long mn = (long long)m * n;
        if (!make_tmap_3d(&tmM, M, TmapType::F32, n, m, batch, (long long)n * 4, mn * 4, 32, kBM) ||
            !make_tmap_3d(&tmG, G, TmapType::BF16, n, m, batch, (long long)n * 2, mn * 2, 64, kBM) ||
            !make_tmap_3d(&tmX, X, TmapType::BF16, n, m, batch, (long long)n * 2, mn * 2, 64, kBM))
            return DION_ERR_CUDA;
        const int tm = (int)cdiv(m, kBM), tn = (int)cdiv(n, kUBN);
        const long long tiles = (long long)tm * tn * batch;
        const int grid = (int)std::min<long long>(tiles, num_sms());
        UpdPArgs ua{m, n, batch, (int)cdiv(rp, kBK), tm, tn, hp, status, tm < tn ? 1 : 0};
        if (ua.kchunks <= 4) {
            static std::atomic<unsigned long long> pattr{0};
            DION_TRY(smem_attr_once((const void*)dion_update_persist_kernel<3, 2>, (int)upd_smem<3, 2>(), pattr));
            DION_TRY(launch("dion_update_tc", dion_update_persist_kernel<3, 2>, dim3(grid), dim3(kUpdThreads), upd_smem<3, 2>(),
                            st, tmPa, tmR, tmQ, tmM, tmG, tmX, ua));
        } else {
            static std::atomic<unsigned long long> pattr_w{0};
            DION_TRY(smem_attr_once((const void*)dion_update_persist_kernel<5, 1>, (int)upd_smem<5, 1>(), pattr_w));
            DION_TRY(launch("dion_update_tc", dion_update_persist_kernel<5, 1>, dim3(grid), dim3(kUpdThreads), upd_smem<5, 1>(),
                            st, tmPa, tmR, tmQ, tmM, tmG, tmX, ua));
        }
    } else {
        static std::atomic<unsigned long long> attr[2] = {{0}, {0}};
        auto k = vec ? dion_update_tc_kernel<true> : dion_update_tc_kernel<false>;
        DION_TRY(smem_attr_once((const void*)k, (int)kUpdSmem, attr[vec]));
        UpdArgs ua{m, n, rp, (int)cdiv(rp, kBK), M, G, X, hp, status};
        DION_TRY(launch("dion_update_tc", k, dim3((unsigned)cdiv(n, kUBN), (unsigned)cdiv(m, kBM), batch), dim3(192),
                        kUpdSmem, st, tmPa, tmR, tmQ, ua));
    }
    return DION_OK;
}

}  // namespace dion
