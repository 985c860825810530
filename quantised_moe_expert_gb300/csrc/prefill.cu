// Prefill path: grouped GEMMs of the experts on the 5th-generation tensor cores.
//
// The expert contraction at large T is a dense GEMM per expert (the "tensor-core
// MoE GEMM with int4-dequant" of the page "POC for qwen3.5 / qwen3.6 support
// optimized for AGX Orin", Phase 9b, there with wmma on sm_87).  Here each CTA
// computes a 128-row weight tile of one expert against up to 128 (gate/up) or
// 256 (down) of the expert's tokens, swap-AB style: weights are the M = 128
// operand, tokens the N operand, so an expert with few tokens still fills the
// MMA's M dimension.
//
// Per K-step (one quantisation group of 64 inputs):
//   - a TMA thread loads the int4 code tile of the weights (128 rows x 32 B),
//     and for the down GEMM the h tile (128-byte swizzle), on an mbarrier;
//   - four dequantising warps turn codes into fp16 w = s*q + b (one rounding)
//     and store them in the 128-byte-swizzled K-major layout the MMA reads;
//     for the gate/up GEMM they also gather the expert's token rows of x
//     with cp.async (16-byte chunks placed at their swizzled positions), one
//     K-step ahead;
//   - one thread issues tcgen05.mma (fp16 in, fp32 accumulate in TMEM) and
//     releases the stage with tcgen05.commit.
// The epilogue reads the accumulators with tcgen05.ld: the gate/up GEMM writes
// h = silu(g) * u as fp16 in expert-sorted row order, the down GEMM adds
// p * y into the fp32 layer accumulator with atomics.
//
// Operand type.  MMA operands are fp16: dequantised weights and the
// intermediate h keep 11 significant bits (bf16 would keep 8, which puts the
// layer output outside the parity tolerance), at the same tensor-core rate.
// x is converted bf16 -> fp16, exact for |x| in [2^-14, 65504].
//
// K order.  Within every 8 consecutive inputs the operands are stored in the
// order (0,4,1,5,2,6,3,7): that is the order in which two bit operations turn
// a 32-bit word of 8 nibbles into four fp16 pairs.  x16 and h are written in
// the same order, so every product still pairs w_j with x_j.
//
// Every wait is bounded; a wait that runs out records MOE_ERR_TIMEOUT, the
// CTA drains its in-flight copies and MMAs, frees its TMEM and returns.
#include <cudaTypedefs.h>

#include <algorithm>

#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace qmoe {
namespace {

using namespace tc;

constexpr int kStages = 3;
constexpr int kThreads = 192;        // warps 0-3 dequant + epilogue, warp 4 TMA, warp 5 MMA
constexpr int kScaleChunk = 32;      // groups of scales staged in shared memory at a time
constexpr long long kDrainLimit = 1ll << 22;

struct G1Params {
    const int32_t *nwork;
    const WorkItem *work;
    const int32_t *offsets;
    const int32_t *perm;
    uint16_t *hs;                      // fp16 [T*k + T, I] (K-permuted), expert-sorted rows
    const uint16_t *x16;               // fp16 [T, H] (K-permuted)
    const uint16_t *gs, *gb, *us, *ub;     // routed gate/up scales, biases [E, I, H/64]
    const uint16_t *sgs, *sgb, *sus, *sub; // shared expert [I, H/64]
    int *status;
    int T, H, I, E, k;
    long long wait_limit;
};

struct G2Params {
    const int32_t *nwork;
    const WorkItem *work;
    const int32_t *offsets;
    const int32_t *perm;
    const uint16_t *p;                 // bf16 [T, k]
    const uint16_t *w_s;               // bf16 [T]
    float *acc;                        // f32 [T, H]
    const uint16_t *ds, *db;           // routed down scales, biases [E, H, I/64]
    const uint16_t *sds, *sdb;         // shared [H, I/64]
    int *status;
    int T, H, I, E, k;
    long long wait_limit;
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk)
{
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// 8 nibbles (inputs 0..7 of a chunk) -> 8 fp16 w = s*q + b in the order (0,4,1,5,2,6,3,7).
__device__ __forceinline__ uint4 dequant8(uint32_t u, __half2 s2, __half2 b2)
{
    const __half2 k1024 = __float2half2_rn(1024.f);
    uint4 o;
    o.x = h2u(__hfma2(__hsub2(u2h((u & 0x000F000Fu) | 0x64006400u), k1024), s2, b2));
    o.y = h2u(__hfma2(__hsub2(u2h(((u >> 4) & 0x000F000Fu) | 0x64006400u), k1024), s2, b2));
    o.z = h2u(__hfma2(__hsub2(u2h(((u >> 8) & 0x000F000Fu) | 0x64006400u), k1024), s2, b2));
    o.w = h2u(__hfma2(__hsub2(u2h(((u >> 12) & 0x000F000Fu) | 0x64006400u), k1024), s2, b2));
    return o;
}

__device__ __forceinline__ __half2 bf16_to_h2(uint16_t b)
{
    return __float2half2_rn(bf16_bits_to_float(b));
}

// Position of input i in the K-permuted storage of its 8-input chunk.
__device__ __forceinline__ int kperm_pos(int i)
{
    const int j = i & 7;
    return (i & ~7) | ((j & 3) << 1) | (j >> 2);
}

__device__ __forceinline__ void set_abort(volatile int *abort, int *status)
{
    *abort = 1;
    record_status(status, MOE_ERR_TIMEOUT);
}

// Stage one chunk of a row's scales and biases (groups [g0, g0 + 32)) into the
// thread-private columns of the shared staging arrays.
__device__ __forceinline__ void stage_scales(uint16_t *dst, const uint16_t *const *src, int nsrc, int row_ok,
                                             size_t row_off, int G, int g0, int r)
{
    for (int a = 0; a < nsrc; ++a)
        for (int g = 0; g < kScaleChunk; ++g) {
            const int gg = g0 + g;
            dst[(a * kScaleChunk + g) * 128 + r] = (row_ok && gg < G) ? src[a][row_off + gg] : (uint16_t)0;
        }
}

// --------------------------------------------------------------- gate/up GEMM
template <int S>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_gateup_kernel(const __grid_constant__ CUtensorMap map_gc, const __grid_constant__ CUtensorMap map_uc,
                       const __grid_constant__ CUtensorMap map_sgc, const __grid_constant__ CUtensorMap map_suc,
                       const G1Params P)
{
    if ((int)blockIdx.y >= __ldg(P.nwork + 1)) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA_g = smem;                         // S x 16 KB
    uint8_t *sA_u = sA_g + S * 16384;             // S x 16 KB
    uint8_t *sB = sA_u + S * 16384;               // S x 16 KB (128 rows x 128 B)
    uint8_t *sC = sB + S * 16384;                 // S x 8 KB (gate codes 4 KB | up codes 4 KB)
    uint16_t *sScale = reinterpret_cast<uint16_t *>(sC + S * 8192);   // [4][32][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sScale + 4 * kScaleChunk * 128);
    uint64_t *full = bars, *afull = bars + S, *empty = bars + 2 * S, *accf = bars + 3 * S, *drain = accf + 1;
    int *s_rows = reinterpret_cast<int *>(drain + 1);     // [128]
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(s_rows + 128);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WorkItem it = P.work[blockIdx.y];
    const bool shared_e = it.expert == P.E;
    const int i0 = blockIdx.x * 128;
    const int ntok = it.ntok;
    const int N = (ntok + 15) & ~15;
    const int H = P.H, I = P.I, G = H / kGroup, nk = G;
    const int pbase = shared_e ? P.T * P.k + it.tok0 : __ldg(P.offsets + it.expert) + it.tok0;

    if (tid < 128) {
        int row = 0;                              // rows past ntok are never read
        if (tid < ntok) {
            if (shared_e) {
                row = it.tok0 + tid;
            } else {
                const int pos = pbase + tid;
                const int f = (pos >= 0 && pos < P.T * P.k) ? __ldg(P.perm + pos) : -1;
                if (f < 0 || f >= P.T * P.k) record_status(P.status, MOE_ERR_DEVICE);
                else row = f / P.k;
            }
        }
        s_rows[tid] = row;
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(s_tmem), 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(afull + s), 128);
            mbar_init(smem_u32(empty + s), 1);
        }
        mbar_init(smem_u32(accf), 1);
        mbar_init(smem_u32(drain), 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long limit = P.wait_limit;

    if (warp == 4) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const CUtensorMap *mg = shared_e ? &map_sgc : &map_gc;
            const CUtensorMap *mu = shared_e ? &map_suc : &map_uc;
            prefetch_map(mg);
            prefetch_map(mu);
            const int wrow = (shared_e ? 0 : it.expert * I) + i0;
            const uint32_t bytes = 8192;
            int issued = 0;
            for (int s = 0; s < nk; ++s) {
                const int st = s % S, rnd = s / S;
                if (s >= S && !mbar_wait(smem_u32(empty + st), (rnd - 1) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    break;
                }
                const uint32_t fb = smem_u32(full + st);
                mbar_arrive_expect_tx(fb, bytes);
                tma_load_2d(smem_u32(sC + st * 8192), mg, s * 32, wrow, fb);
                tma_load_2d(smem_u32(sC + st * 8192 + 4096), mu, s * 32, wrow, fb);
                issued = s + 1;
            }
            if (*s_abort) {
                // drain: every issued stage's copies must land before the CTA exits
                for (int s = (issued > S ? issued - S : 0); s < issued; ++s)
                    mbar_wait(smem_u32(full + s % S), (s / S) & 1, kDrainLimit, nullptr);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_m128((uint32_t)N);
            bool ok = true;
            for (int s = 0; s < nk && ok; ++s) {
                const int st = s % S, rnd = s / S;
                if (!mbar_wait(smem_u32(afull + st), rnd & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t ag = smem_u32(sA_g + st * 16384), au = smem_u32(sA_u + st * 16384);
                const uint32_t bb = smem_u32(sB + st * 16384);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acc = (s | kk) != 0;
                    mma_f16(tmem, desc_sw128(ag + kk * 32), desc_sw128(bb + kk * 32), idesc, acc);
                    mma_f16(tmem + 128, desc_sw128(au + kk * 32), desc_sw128(bb + kk * 32), idesc, acc);
                }
                mma_commit(smem_u32(empty + st));
            }
            if (ok) mma_commit(smem_u32(accf));
            // every MMA this thread issued completes before TMEM is freed, on every path
            mma_commit(smem_u32(drain));
            mbar_wait(smem_u32(drain), 0, kDrainLimit, nullptr);
        }
    } else {
        // ------------------------------------------------ dequant (thread = weight row) + token rows
        const int r = tid;
        const int row = i0 + r;
        const bool row_ok = row < I;
        const size_t soff = (size_t)(shared_e ? 0 : it.expert) * I * G + (size_t)row * G;
        const uint16_t *srcs[4] = {shared_e ? P.sgs : P.gs, shared_e ? P.sgb : P.gb, shared_e ? P.sus : P.us,
                                   shared_e ? P.sub : P.ub};
        // token rows: thread copies 16-byte chunk (tid & 7) of tile rows (tid >> 3) + 16 i
        const int bchunk = tid & 7, brow0 = tid >> 3;
        auto issue_b = [&](int ks) {
            uint8_t *dst = sB + (ks % S) * 16384;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int n = brow0 + 16 * i;
                if (n < ntok) {
                    const uint16_t *src = P.x16 + (size_t)s_rows[n] * H + ks * 64 + bchunk * 8;
                    cp_async16(smem_u32(dst + swz128(n, bchunk)), src);
                }
            }
            cp_async_commit();
        };
        bool ok = true;
        issue_b(0);
        for (int s = 0; s < nk; ++s) {
            const int st = s % S, rnd = s / S;
            if (s % kScaleChunk == 0) stage_scales(sScale, srcs, 4, row_ok, soff, G, s, r);
            if (s + 1 < nk) {
                const int sn = s + 1;
                if (sn >= S && !mbar_wait(smem_u32(empty + sn % S), (sn / S - 1) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                issue_b(sn);
            } else {
                cp_async_commit();
            }
            if (!mbar_wait(smem_u32(full + st), rnd & 1, limit, s_abort)) {
                set_abort(s_abort, P.status);
                ok = false;
                break;
            }
            const int gi = s % kScaleChunk;
            const __half2 sg = bf16_to_h2(sScale[(0 * kScaleChunk + gi) * 128 + r]);
            const __half2 bg = bf16_to_h2(sScale[(1 * kScaleChunk + gi) * 128 + r]);
            const __half2 su = bf16_to_h2(sScale[(2 * kScaleChunk + gi) * 128 + r]);
            const __half2 bu = bf16_to_h2(sScale[(3 * kScaleChunk + gi) * 128 + r]);
            const uint4 *cg = reinterpret_cast<const uint4 *>(sC + st * 8192 + r * 32);
            const uint4 *cu = reinterpret_cast<const uint4 *>(sC + st * 8192 + 4096 + r * 32);
            const uint4 g0 = cg[0], g1 = cg[1], u0 = cu[0], u1 = cu[1];
            const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const uint32_t uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            uint8_t *ag = sA_g + st * 16384;
            uint8_t *au = sA_u + st * 16384;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                *reinterpret_cast<uint4 *>(ag + swz128(r, c)) = dequant8(gw[c], sg, bg);
                *reinterpret_cast<uint4 *>(au + swz128(r, c)) = dequant8(uw[c], su, bu);
            }
            cp_async_wait_1();               // this K-step's token rows have landed
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(afull + st));
        }
        cp_async_wait_all();
        // ------------------------------------------------ epilogue: h = silu(g) * u
        if (ok && mbar_wait(smem_u32(accf), 0, limit, s_abort)) {
            tc_fence_after();
            const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
            const int erow = i0 + warp * 32 + lane;
            const int hcol = kperm_pos(erow);
            for (int n0 = 0; n0 < N; n0 += 16) {
                uint32_t gv[16], uv[16];
                tmem_ld16(tmem + lane_base + n0, gv);
                tmem_ld16(tmem + lane_base + 128 + n0, uv);
                tmem_ld_wait();
                if (erow < I) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = n0 + j;
                        if (n < ntok) {
                            const float g = __uint_as_float(gv[j]), u = __uint_as_float(uv[j]);
                            const float hv = g / (1.f + __expf(-g)) * u;
                            P.hs[(size_t)(pbase + n) * I + hcol] = __half_as_ushort(__float2half_rn(hv));
                        }
                    }
                }
            }
        } else if (ok) {
            set_abort(s_abort, P.status);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// --------------------------------------------------------------- down GEMM
template <int S>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_down_kernel(const __grid_constant__ CUtensorMap map_dc, const __grid_constant__ CUtensorMap map_sdc,
                     const __grid_constant__ CUtensorMap map_h, const G2Params P)
{
    if ((int)blockIdx.y >= __ldg(P.nwork + 2)) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                           // S x 16 KB
    uint8_t *sB = sA + S * 16384;                 // S x 32 KB (256 rows x 128 B)
    uint8_t *sC = sB + S * 32768;                 // S x 4 KB
    uint16_t *sScale = reinterpret_cast<uint16_t *>(sC + S * 4096);   // [2][32][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sScale + 2 * kScaleChunk * 128);
    uint64_t *full = bars, *afull = bars + S, *empty = bars + 2 * S, *accf = bars + 3 * S, *drain = accf + 1;
    int *s_tok = reinterpret_cast<int *>(drain + 1);           // [256]
    float *s_w = reinterpret_cast<float *>(s_tok + 256);       // [256]
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(s_w + 256);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WorkItem it = P.work[blockIdx.y];
    const bool shared_e = it.expert == P.E;
    const int h0 = blockIdx.x * 128;
    const int ntok = it.ntok;
    const int N = (ntok + 15) & ~15;
    const int nbox = (N + 31) / 32;
    const int H = P.H, I = P.I, GI = I / kGroup, nk = GI;
    const int pbase = shared_e ? P.T * P.k + it.tok0 : __ldg(P.offsets + it.expert) + it.tok0;

    for (int n = tid; n < 256; n += blockDim.x) {
        int t = -1;
        float wgt = 0.f;
        if (n < ntok) {
            if (shared_e) {
                t = it.tok0 + n;
                wgt = bf16_bits_to_float(P.w_s[t]);
            } else {
                const int pos = pbase + n;
                const int f = (pos >= 0 && pos < P.T * P.k) ? __ldg(P.perm + pos) : -1;
                if (f < 0 || f >= P.T * P.k) {
                    record_status(P.status, MOE_ERR_DEVICE);
                } else {
                    t = f / P.k;
                    wgt = bf16_bits_to_float(P.p[f]);
                }
            }
        }
        s_tok[n] = t;
        s_w[n] = wgt;
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(s_tmem), 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(afull + s), 128);
            mbar_init(smem_u32(empty + s), 1);
        }
        mbar_init(smem_u32(accf), 1);
        mbar_init(smem_u32(drain), 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long limit = P.wait_limit;

    if (warp == 4) {
        if (lane == 0) {
            const CUtensorMap *md = shared_e ? &map_sdc : &map_dc;
            prefetch_map(md);
            prefetch_map(&map_h);
            const int wrow = (shared_e ? 0 : it.expert * H) + h0;
            const uint32_t bytes = 4096 + (uint32_t)nbox * 32 * 128;
            int issued = 0;
            for (int s = 0; s < nk; ++s) {
                const int st = s % S, rnd = s / S;
                if (s >= S && !mbar_wait(smem_u32(empty + st), (rnd - 1) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    break;
                }
                const uint32_t fb = smem_u32(full + st);
                mbar_arrive_expect_tx(fb, bytes);
                tma_load_2d(smem_u32(sC + st * 4096), md, s * 32, wrow, fb);
                for (int q = 0; q < nbox; ++q)
                    tma_load_2d(smem_u32(sB + st * 32768 + q * 4096), &map_h, s * 64, pbase + q * 32, fb);
                issued = s + 1;
            }
            if (*s_abort)
                for (int s = (issued > S ? issued - S : 0); s < issued; ++s)
                    mbar_wait(smem_u32(full + s % S), (s / S) & 1, kDrainLimit, nullptr);
        }
    } else if (warp == 5) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_m128((uint32_t)N);
            bool ok = true;
            for (int s = 0; s < nk; ++s) {
                const int st = s % S, rnd = s / S;
                if (!mbar_wait(smem_u32(full + st), rnd & 1, limit, s_abort) ||
                    !mbar_wait(smem_u32(afull + st), rnd & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t aa = smem_u32(sA + st * 16384), bb = smem_u32(sB + st * 32768);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(tmem, desc_sw128(aa + kk * 32), desc_sw128(bb + kk * 32), idesc, (s | kk) != 0);
                mma_commit(smem_u32(empty + st));
            }
            if (ok) mma_commit(smem_u32(accf));
            // every MMA this thread issued completes before TMEM is freed, on every path
            mma_commit(smem_u32(drain));
            mbar_wait(smem_u32(drain), 0, kDrainLimit, nullptr);
        }
    } else {
        const int r = tid;
        const int row = h0 + r;
        const bool row_ok = row < H;
        const size_t soff = (size_t)(shared_e ? 0 : it.expert) * H * GI + (size_t)row * GI;
        const uint16_t *srcs[2] = {shared_e ? P.sds : P.ds, shared_e ? P.sdb : P.db};
        bool ok = true;
        for (int s = 0; s < nk; ++s) {
            const int st = s % S, rnd = s / S;
            if (s % kScaleChunk == 0) stage_scales(sScale, srcs, 2, row_ok, soff, GI, s, r);
            if (!mbar_wait(smem_u32(full + st), rnd & 1, limit, s_abort)) {
                set_abort(s_abort, P.status);
                ok = false;
                break;
            }
            const int gi = s % kScaleChunk;
            const __half2 sd = bf16_to_h2(sScale[(0 * kScaleChunk + gi) * 128 + r]);
            const __half2 bd = bf16_to_h2(sScale[(1 * kScaleChunk + gi) * 128 + r]);
            const uint4 *cd = reinterpret_cast<const uint4 *>(sC + st * 4096 + r * 32);
            const uint4 c0 = cd[0], c1 = cd[1];
            const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint8_t *aa = sA + st * 16384;
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(aa + swz128(r, c)) = dequant8(cw[c], sd, bd);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(afull + st));
        }
        // ------------------------------------------------ epilogue: acc[t, row] += w * y
        if (ok && mbar_wait(smem_u32(accf), 0, limit, s_abort)) {
            tc_fence_after();
            const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
            const int erow = h0 + warp * 32 + lane;
            for (int n0 = 0; n0 < N; n0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + lane_base + n0, v);
                tmem_ld_wait();
                if (erow < H) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = n0 + j;
                        const int t = n < ntok ? s_tok[n] : -1;
                        if (t >= 0) atomicAdd(P.acc + (size_t)t * H + erow, s_w[n] * __uint_as_float(v[j]));
                    }
                }
            }
        } else if (ok) {
            set_abort(s_abort, P.status);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// x (bf16 [T, H]) -> x16 (fp16 [T, H], K-permuted within chunks of 8)
__global__ void convert_x_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ x16, size_t nchunks)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nchunks; i += (size_t)gridDim.x * blockDim.x) {
        const uint4 v = x[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float f[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = __uint_as_float(w[j] << 16);
            f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
        uint4 o;
        o.x = h2u(__floats2half2_rn(f[0], f[4]));
        o.y = h2u(__floats2half2_rn(f[1], f[5]));
        o.z = h2u(__floats2half2_rn(f[2], f[6]));
        o.w = h2u(__floats2half2_rn(f[3], f[7]));
        x16[i] = o;
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2D row-major map: inner extent `cols` elements, `rows` rows, box {bc, br}.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, uint64_t cols, uint64_t rows,
              uint32_t bc, uint32_t br, CUtensorMapSwizzle swz)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * (uint64_t)esize};
    cuuint32_t box[2] = {bc, br};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t g1_smem() { return 1024 + kStages * (16384 * 3 + 8192) + 4 * kScaleChunk * 128 * 2 + 8 * (3 * kStages + 2) + 128 * 4 + 16; }
size_t g2_smem() { return 1024 + kStages * (16384 + 32768 + 4096) + 2 * kScaleChunk * 128 * 2 + 8 * (3 * kStages + 2) + 512 * 4 + 16; }

}  // namespace

cudaError_t launch_prefill_experts(const PrefillArgs &a, cudaStream_t st)
{
    const int H = a.H, I = a.I, E = a.E, T = a.T, k = a.k;
    // x -> fp16, K-permuted
    {
        const size_t n = (size_t)T * H / 8;
        const unsigned grid = (unsigned)std::min<size_t>((n + 255) / 256, 152 * 8);
        convert_x_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4 *>(a.x), reinterpret_cast<uint4 *>(a.x16),
                                               n);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaSuccess;
    if (a.acc_zero && (e = launch_zero(a.acc, (size_t)T * H, st)) != cudaSuccess) return e;

    CUtensorMap mgc, muc, msgc, msuc, mdc, msdc, mh;
    const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE, sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int ns = a.has_shared ? 1 : 0;
    bool ok = make_map(&mgc, a.gate.codes, u8, 1, H / 2, (uint64_t)E * I, 32, 128, none) &&
              make_map(&muc, a.up.codes, u8, 1, H / 2, (uint64_t)E * I, 32, 128, none) &&
              make_map(&mdc, a.down.codes, u8, 1, I / 2, (uint64_t)E * H, 32, 128, none) &&
              make_map(&mh, a.hs, f16, 2, I, (uint64_t)T * k + (uint64_t)T, 64, 32, sw128);
    if (ns)
        ok = ok && make_map(&msgc, a.s_gate.codes, u8, 1, H / 2, I, 32, 128, none) &&
             make_map(&msuc, a.s_up.codes, u8, 1, H / 2, I, 32, 128, none) &&
             make_map(&msdc, a.s_down.codes, u8, 1, I / 2, H, 32, 128, none);
    else {
        msgc = mgc;
        msuc = muc;
        msdc = mdc;
    }
    if (!ok) return cudaErrorInvalidValue;

    G1Params p1{};
    p1.nwork = a.nwork;
    p1.work = a.work_g1;
    p1.offsets = a.offsets;
    p1.perm = a.perm;
    p1.hs = a.hs;
    p1.x16 = a.x16;
    p1.gs = a.gate.scales;
    p1.gb = a.gate.biases;
    p1.us = a.up.scales;
    p1.ub = a.up.biases;
    p1.sgs = a.s_gate.scales;
    p1.sgb = a.s_gate.biases;
    p1.sus = a.s_up.scales;
    p1.sub = a.s_up.biases;
    p1.status = a.status;
    p1.T = T;
    p1.H = H;
    p1.I = I;
    p1.E = E;
    p1.k = k;
    p1.wait_limit = a.wait_limit;
    const size_t s1 = g1_smem();
    cudaFuncSetAttribute(gemm_gateup_kernel<kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
    gemm_gateup_kernel<kStages><<<dim3((I + 127) / 128, a.max_w1), kThreads, s1, st>>>(mgc, muc, msgc, msuc, p1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    G2Params p2{};
    p2.nwork = a.nwork;
    p2.work = a.work_g2;
    p2.offsets = a.offsets;
    p2.perm = a.perm;
    p2.p = a.p;
    p2.w_s = a.w_s;
    p2.acc = a.acc;
    p2.ds = a.down.scales;
    p2.db = a.down.biases;
    p2.sds = a.s_down.scales;
    p2.sdb = a.s_down.biases;
    p2.status = a.status;
    p2.T = T;
    p2.H = H;
    p2.I = I;
    p2.E = E;
    p2.k = k;
    p2.wait_limit = a.wait_limit;
    const size_t s2 = g2_smem();
    cudaFuncSetAttribute(gemm_down_kernel<kStages>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
    gemm_down_kernel<kStages><<<dim3((H + 127) / 128, a.max_w2), kThreads, s2, st>>>(mdc, msdc, mh, p2);
    return cudaGetLastError();
}

}  // namespace qmoe
