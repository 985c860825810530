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
// Both kernels are persistent (one CTA per SM looping over tiles) and warp
// specialised.  Per K-step (one quantisation group of 64 inputs):
//   - a TMA thread streams the int4 code tile of the weights (128 rows x 32 B)
//     through a ring of code stages;
//   - the token operand arrives in its own, deeper ring: for the gate/up GEMM a
//     loader warp gathers the expert's rows of x with cp.async (16-byte chunks
//     placed at their 128-byte-swizzled positions), for the down GEMM a second
//     TMA thread loads the h tile;
//   - eight dequantising warps turn codes into fp16 w = s*q + b (one rounding)
//     and store them in the swizzled K-major layout the MMA reads;
//   - one thread issues tcgen05.mma (fp16 in, fp32 accumulate in TMEM) and
//     releases each stage with tcgen05.commit.
// Epilogue warps read the accumulators with tcgen05.ld: the gate/up GEMM writes
// h = silu(g) * u as fp16 in expert-sorted row order; the down GEMM, from the
// other half of TMEM while the next tile accumulates, writes each slot's expert
// output y_e (fp32) once with bulk stores, and the slots of every token are
// summed afterwards in a fixed order (the pick weights applied there).
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
// NVFP4 experts (E2M1 codes, an E4M3 scale per 16 inputs, an fp32 scale per
// matrix).  The code tiles are those of the 4-bit codes.  A K-step's four block
// scales of a row arrive through the same private scale buffer (4 bytes a group
// in place of the bf16 scale and bias), each code word is expanded by the
// hardware E2M1 -> fp16 conversion and multiplied by its block's scale in fp16
// (exact: at most 6 significant bits in [2^-10, 2688]), and the matrix scale is
// applied to the fp32 accumulators in the epilogues.
//
// Every wait is bounded; a wait that runs out records MOE_ERR_TIMEOUT, the
// CTA drains its in-flight copies and MMAs, frees its TMEM and returns.
#include <algorithm>

#include "kernels.cuh"
#include "nvfp4.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace qmoe {
namespace {

using namespace tc;

// Stage counts of the three rings of each GEMM: dequantised weights (A), token
// operand (B) and code tiles.  B runs deepest: its loads come from L2 / HBM with
// a latency of several K-steps of MMA.  A code stage holds one K-step (64 inputs)
// of 128 rows: 32 bytes a row for 4-bit codes, 64 for 8-bit codes, so the 8-bit
// rings have half the stages in the same bytes.
constexpr int kStagesA1 = 4, kStagesB1 = 8, kCodeStages1 = 6;   // gate/up: A in TMEM (64 columns), 16 KB, 8 KB per stage
constexpr int kStagesA2 = 3, kStagesB2 = 3, kCodeStages2 = 6;   // down:    16 KB, 32 KB, 4 KB per stage
constexpr int kCodeStages1B8 = 3, kCodeStages2B8 = 3;           // 8-bit codes: 16 KB / 8 KB per stage

// Bytes of one row's codes per K-step, and of one code stage of each GEMM (gate | up; down).
constexpr int cbits(int bits) { return bits == kNvfp4 ? 4 : bits; }   // code width of the args' code field
constexpr int code_row_bytes(int bits) { return 8 * cbits(bits); }
constexpr int code_stage1(int bits) { return 2 * 128 * code_row_bytes(bits); }
constexpr int code_stage2(int bits) { return 128 * code_row_bytes(bits); }
constexpr int kRedCols = 16, kRedBufs = 2;   // down epilogue: columns per store chunk, chunk buffers per team
// Warp roles of the down GEMM: 0-7 dequantise, 8 TMA, 9 MMA, 10-17 epilogue (two teams of four warps,
// one warp per TMEM lane quarter, taking the 16-column chunks of a tile in turn).
constexpr int kDequantThreads = 256;
constexpr int kWarpTma = 8, kWarpMma = 9, kWarpEpi = 10, kEpiTeams2 = 2;
constexpr int kThreads = 32 * (kWarpEpi + 4 * kEpiTeams2);     // down GEMM: 576
// Gate/up GEMM: warps 0-15 dequantise (0-7 the even K-steps, 8-15 the odd ones, so two
// steps of each row are in flight), 16 TMA, 17 MMA, 18-25 epilogue (two per TMEM lane quarter:
// the epilogue holds the single accumulator pair, so the MMAs of the next tile wait for it),
// and two token-row loader warps (26, 27) that take the K-steps in turn, each with kLoaderDepth of its
// steps in flight.
constexpr int kDequantWarps1 = 16, kStepWarps1 = 8;
constexpr int kWarpTma1 = 16, kWarpMma1 = 17, kWarpEpi1 = 18, kEpiWarps1 = 8;
constexpr int kWarpLoader1 = kWarpEpi1 + kEpiWarps1, kLoaderWarps1 = 2, kLoaderDepth = 2;
constexpr int kThreads1 = 32 * (kWarpLoader1 + kLoaderWarps1);  // 896
constexpr int kScaleChunk1 = 8;                                 // gate/up: groups per scale chunk
constexpr long long kDrainLimit = 1ll << 22;
constexpr uint32_t kTmemA1 = 256;   // gate/up GEMM: accumulators in TMEM columns [0, 256), A stages from 256

struct G1Params {
    const int32_t *nwork;
    const WorkItem *work;
    const int32_t *offsets;
    const int32_t *perm;
    uint16_t *hs;                      // fp16 [T*k + T, I] (K-permuted), expert-sorted rows: h' = h 2^-2e
    const uint16_t *x16;               // fp16 [T, H] (K-permuted): x' = x 2^-e
    const int *xe;                     // i32 [T]: e of each token
    float *h_out;                      // f32 [T*k + T, I] h per slot (stage output), or null
    const uint8_t *gc, *uc, *sgc, *suc;    // int4 codes (routed [E, I, H/2], shared [I, H/2]), for L2 prefetch
    const uint16_t *gs, *gb, *us, *ub;     // routed gate/up scales, biases [E, I, H/64]
    const uint16_t *sgs, *sgb, *sus, *sub; // shared expert [I, H/64]
    const float *ggs, *ugs, *sggs, *sugs;  // NVFP4: matrix scales (routed [E], shared [1])
    int *status;
    int T, H, I, E, k;
    int async_scales;                  // 1: scale rows are 16-byte aligned (H % 512 == 0), fetched with cp.async
    long long wait_limit;
};

struct G2Params {
    const int32_t *nwork;
    const WorkItem *work;
    const int32_t *offsets;
    const int32_t *perm;
    const int *xe;                     // i32 [T]: e of each token (the h tile holds h 2^-2e)
    float *yslot;                      // f32 [T*k + T, H]: each slot's expert output before its pick weight, rows
                                       // in expert-sorted position order (the rows of the h tiles)
    const uint8_t *dc, *sdc;           // int4 codes (routed [E, H, I/2], shared [H, I/2]), for L2 prefetch
    const uint16_t *ds, *db;           // routed down scales, biases [E, H, I/64]
    const uint16_t *sds, *sdb;         // shared [H, I/64]
    const float *dgs, *sdgs;           // NVFP4: matrix scales (routed [E], shared [1])
    int *status;
    int T, H, I, E, k;
    int async_scales;                  // 1: scale rows are 16-byte aligned (I % 512 == 0), fetched with cp.async
    long long wait_limit;
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk)
{
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// 8 nibbles (inputs 0..7 of a chunk) -> 8 fp16 w = s*q + b in the order (0,4,1,5,2,6,3,7).
// The low nibble of each byte, ORed into the mantissa of 1024.0, gives 1024 + q; the high
// nibble masked in place gives 1024 + 16 q, and s16 = s / 16 (a power-of-two division,
// exact) makes (16 q) * s16 = q * s: one shift per word instead of three.  Every weight is
// the exact s * q + b rounded once to fp16.
__device__ __forceinline__ uint4 dequant8(uint32_t u, __half2 s2, __half2 s16, __half2 b2)
{
    const __half2 k1024 = __float2half2_rn(1024.f);
    const uint32_t v = u >> 8;
    uint4 o;
    o.x = h2u(__hfma2(__hsub2(u2h((u & 0x000F000Fu) | 0x64006400u), k1024), s2, b2));
    o.y = h2u(__hfma2(__hsub2(u2h((u & 0x00F000F0u) | 0x64006400u), k1024), s16, b2));
    o.z = h2u(__hfma2(__hsub2(u2h((v & 0x000F000Fu) | 0x64006400u), k1024), s2, b2));
    o.w = h2u(__hfma2(__hsub2(u2h((v & 0x00F000F0u) | 0x64006400u), k1024), s16, b2));
    return o;
}

__device__ __forceinline__ __half2 bf16_to_h2(uint16_t b)
{
    return __float2half2_rn(bf16_bits_to_float(b));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// 8 byte codes (u0: inputs 0-3, u1: inputs 4-7 of a chunk) -> 8 fp16 w = s*q + b in the same order
// (0,4,1,5,2,6,3,7).  Each byte pair is moved into the mantissas of two 1024.0: 1024 + q is exact for
// q < 1024, the subtraction of 1024 is exact, and w is the exact s * q + b rounded once to fp16.
__device__ __forceinline__ uint4 dequant8_b8(uint32_t u0, uint32_t u1, __half2 s2, __half2 b2)
{
    const __half2 k1024 = __float2half2_rn(1024.f);
    auto one = [&](uint32_t sel) {
        return h2u(__hfma2(__hsub2(u2h((prmt(u0, u1, sel) & 0x00FF00FFu) | 0x64006400u), k1024), s2, b2));
    };
    uint4 o;
    o.x = one(0x4400u);
    o.y = one(0x5511u);
    o.z = one(0x6622u);
    o.w = one(0x7733u);
    return o;
}

// 8-bit code tiles arrive with the 64-byte swizzle (rows of 64 bytes): 16-byte chunk c of row r sits
// at chunk c ^ ((r >> 1) & 3), so the 8 rows that one quarter-warp reads cover all 32 banks.
__device__ __forceinline__ uint32_t swz64(int row, int chunk)
{
    return (uint32_t)(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
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

// Named barrier `id` over `count` threads.  The non-aligned form: a warp may reach it with its
// lanes apart (after a branch taken by one lane), and each warp is brought back together first.
__device__ __forceinline__ void named_bar(int id, int count)
{
    __syncwarp();
    asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier `id` over `count` threads that also ORs a predicate: every
// participant gets the same answer, so a group of warps stops together.
__device__ __forceinline__ bool bar_any(int id, int count, bool pred)
{
    __syncwarp();
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Tile tau of a grouped GEMM: work item tau / MB, weight-row block tau % MB.
struct TileInfo {
    int expert, tok0, ntok, mb, pbase;
    bool shared_e;
};

__device__ __forceinline__ TileInfo tile_info(const WorkItem *work, const int32_t *offsets, int tau, int MB, int E,
                                              int Tk)
{
    const WorkItem it = work[tau / MB];
    TileInfo ti;
    ti.expert = it.expert;
    ti.tok0 = it.tok0;
    ti.ntok = it.ntok;
    ti.mb = tau % MB;
    ti.shared_e = it.expert == E;
    ti.pbase = ti.shared_e ? Tk + it.tok0 : __ldg(offsets + it.expert) + it.tok0;
    return ti;
}

// Asks L2 for `bytes` contiguous bytes in 32 KB pieces (16-byte multiples, 16-byte aligned).
__device__ __forceinline__ void prefetch_rows(const void *p, uint32_t bytes)
{
    const uint8_t *b = static_cast<const uint8_t *>(p);
    for (uint32_t off = 0; off < bytes; off += 32768u) prefetch_l2_bulk(b + off, bytes - off < 32768u ? bytes - off : 32768u);
}

// --------------------------------------------------------------- gate/up GEMM
//
// Persistent: one CTA per SM loops over tiles tau = blockIdx.x + i * gridDim.x.
// Roles (constants above): the dequantising warps turn code tiles into A stages in tensor
// memory; one thread streams code tiles with TMA through a ring of CS stages and asks L2
// for the next tile in bulk; one thread issues the MMAs (A from tensor memory, B from
// shared memory); the epilogue warps turn the accumulators into h; the loader warps
// gather the token rows of x with cp.async into a ring of SB stages.
// Tensor memory: gate and up accumulators in columns [0, 256) (one buffer, so a tile's
// first MMAs wait for the previous epilogue's reads), A stages from column 256.
// BITS: expert code width (4 or 8).
template <int S, int SB, int CS, int BITS>
__global__ void __launch_bounds__(kThreads1, 1)
    gemm_gateup_kernel(const __grid_constant__ CUtensorMap map_gc, const __grid_constant__ CUtensorMap map_uc,
                       const __grid_constant__ CUtensorMap map_sgc, const __grid_constant__ CUtensorMap map_suc,
                       const G1Params P)
{
    const int H = P.H, I = P.I, G = H / kGroup, nk = G, MB = (I + 127) / 128, Tk = P.T * P.k;
    constexpr int CB = code_row_bytes(BITS), CST = code_stage1(BITS);
    const size_t crow = (size_t)H * cbits(BITS) / 8;     // bytes of one weight row's codes
    const int ntiles = __ldg(P.nwork + 3) * MB;          // the big items lead the list
    // This grid may start while the small-tile gate/up GEMM still runs (programmatic
    // dependent launch): it reads nothing that grid writes, and every CTA waits for that
    // grid before it exits, so the kernels after both see all of h.
    if ((int)blockIdx.x >= ntiles) {
        pdl_wait();
        return;
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);
    uint8_t *sB = smem;                           // SB x 16 KB (128 token rows x 128 B)
    uint8_t *sC = sB + SB * 16384;                // CS x CST (gate codes | up codes)
    uint16_t *sScale = reinterpret_cast<uint16_t *>(sC + CS * CST);    // [dequant thread][2][2][kScaleChunk1]
    int *s_col = reinterpret_cast<int *>(sScale + kDequantWarps1 * 32 * 4 * kScaleChunk1);   // [2][e 128 | slot 128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_col + 2 * 256);
    uint64_t *cfull = bars, *cempty = cfull + CS, *afull = cempty + CS, *aempty = afull + S;
    uint64_t *bfull = aempty + S, *bempty = bfull + SB;
    uint64_t *tfull = bempty + SB, *tempty = tfull + 2, *drain = tempty + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == kWarpMma1) {
        tmem_alloc(smem_u32(s_tmem), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < CS; ++s) {
            mbar_init(smem_u32(cfull + s), 1);
            mbar_init(smem_u32(cempty + s), kStepWarps1);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(afull + s), kStepWarps1);
            mbar_init(smem_u32(aempty + s), 1);
        }
        for (int s = 0; s < SB; ++s) {
            mbar_init(smem_u32(bfull + s), 32);           // the lanes of the step's loader warp
            mbar_init(smem_u32(bempty + s), 1);
        }
        mbar_init(smem_u32(tfull), 1);
        mbar_init(smem_u32(tempty), 32 * kEpiWarps1);
        mbar_init(smem_u32(drain), 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long limit = P.wait_limit;

    if (warp >= kWarpLoader1) {
        // ------------------------------------------------ token rows of x (cp.async gather)
        // The loader warps take the K-steps in turn (warp w: steps q = w mod kLoaderWarps1),
        // each keeping kLoaderDepth of its own steps in flight; lane l gathers rows l, l + 32,
        // l + 64 and l + 96 of the tile.  Step q's rows go into stage q % SB once the MMAs of
        // step q - SB are done, and each lane arrives on the stage's full barrier as soon as
        // its own copies of that step have landed.
        const int lw = warp - kWarpLoader1;
        int q = 0, q_last = -1, pending = 0;                  // pending: issued, not yet arrived
        bool ok = true;
        for (int tau = blockIdx.x; tau < ntiles && ok; tau += gridDim.x) {
            const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
            const uint16_t *src[4];                           // rows past ntok are never read
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = lane + 32 * j;
                src[j] = nullptr;
                if (n < ti.ntok) {
                    int row = -1;
                    if (ti.shared_e) {
                        row = ti.tok0 + n;
                    } else {
                        const int pos = ti.pbase + n;
                        const int f = (pos >= 0 && pos < Tk) ? __ldg(P.perm + pos) : -1;
                        if (f < 0 || f >= Tk) record_status(P.status, MOE_ERR_DEVICE);
                        else row = f / P.k;
                    }
                    if (row >= 0) src[j] = P.x16 + (size_t)row * H;
                }
            }
            for (int s = 0; s < nk; ++s, ++q) {
                if (q % kLoaderWarps1 != lw) continue;
                const int st = q % SB;
                if (q >= SB && !mbar_wait(smem_u32(bempty + st), (q / SB - 1) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                uint8_t *dst = sB + st * 16384;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (src[j]) {
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            cp_async16(smem_u32(dst + swz128(lane + 32 * j, c)), src[j] + s * 64 + c * 8);
                    }
                cp_async_commit();
                q_last = q;
                if (++pending == kLoaderDepth) {              // the oldest of this warp's steps has landed
                    cp_async_wait_group<kLoaderDepth - 1>();
                    fence_proxy_async_smem();
                    mbar_arrive(smem_u32(bfull + (q - (kLoaderDepth - 1) * kLoaderWarps1) % SB));
                    --pending;
                }
            }
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        for (int d = pending - 1; d >= 0; --d) mbar_arrive(smem_u32(bfull + (q_last - d * kLoaderWarps1) % SB));
    } else if (warp == kWarpTma1) {
        // ------------------------------------------------ code tiles (TMA)
        if (lane == 0) {
            prefetch_map(&map_gc);
            prefetch_map(&map_uc);
            prefetch_map(&map_sgc);
            prefetch_map(&map_suc);
            // The code boxes are 32 (64) bytes of 128 rows 1 KB (2 KB) apart: fetched from DRAM
            // piece by piece they would cost a DRAM burst each.  A tile's rows are contiguous, so
            // the whole tile (codes, scales, biases) is requested from L2 in bulk one tile ahead.
            auto prefetch_tile = [&](int tp) {
                if (tp >= ntiles) return;
                const TileInfo t2 = tile_info(P.work, P.offsets, tp, MB, P.E, Tk);
                const int rows = min(128, I - t2.mb * 128);
                const size_t wrow = (size_t)(t2.shared_e ? 0 : t2.expert * I) + t2.mb * 128;
                prefetch_rows((t2.shared_e ? P.sgc : P.gc) + wrow * crow, (uint32_t)(rows * crow));
                prefetch_rows((t2.shared_e ? P.suc : P.uc) + wrow * crow, (uint32_t)(rows * crow));
                // scale bytes of a row: bf16 scale (and bias) per group, or NVFP4's 4 E4M3 bytes per group
                constexpr int kSb = BITS == kNvfp4 ? 4 : 2;
                const uint32_t sb = (uint32_t)rows * G * kSb;
                const size_t so = wrow * G * kSb;
                prefetch_rows(reinterpret_cast<const uint8_t *>(t2.shared_e ? P.sgs : P.gs) + so, sb);
                prefetch_rows(reinterpret_cast<const uint8_t *>(t2.shared_e ? P.sus : P.us) + so, sb);
                if constexpr (BITS != kNvfp4) {           // NVFP4 has no biases
                    prefetch_rows((t2.shared_e ? P.sgb : P.gb) + wrow * G, sb);
                    prefetch_rows((t2.shared_e ? P.sub : P.ub) + wrow * G, sb);
                }
            };
            prefetch_tile(blockIdx.x);
            int q = 0;
            bool ok = true;
            for (int tau = blockIdx.x; tau < ntiles && ok; tau += gridDim.x) {
                const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
                prefetch_tile(tau + gridDim.x);
                const CUtensorMap *mg = ti.shared_e ? &map_sgc : &map_gc;
                const CUtensorMap *mu = ti.shared_e ? &map_suc : &map_uc;
                const int wrow = (ti.shared_e ? 0 : ti.expert * I) + ti.mb * 128;
                for (int s = 0; s < nk; ++s, ++q) {
                    const int cs = q % CS;
                    if (q >= CS && !mbar_wait(smem_u32(cempty + cs), (q / CS - 1) & 1, limit, s_abort)) {
                        set_abort(s_abort, P.status);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(cfull + cs);
                    mbar_arrive_expect_tx(fb, CST);
                    tma_load_2d(smem_u32(sC + cs * CST), mg, s * CB, wrow, fb);
                    tma_load_2d(smem_u32(sC + cs * CST + CST / 2), mu, s * CB, wrow, fb);
                }
            }
            if (!ok || *s_abort)   // every issued copy lands before the CTA exits
                for (int d = (q > CS ? q - CS : 0); d < q; ++d)
                    mbar_wait(smem_u32(cfull + d % CS), (d / CS) & 1, kDrainLimit, nullptr);
        }
    } else if (warp == kWarpMma1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int q = 0, i = 0;
            bool ok = true;
            for (int tau = blockIdx.x; tau < ntiles && ok; tau += gridDim.x, ++i) {
                const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
                const int N = (ti.ntok + 15) & ~15;
                const uint32_t idesc = idesc_f16_m128((uint32_t)N);
                // one accumulator pair: the epilogue of the previous tile has read it
                if (i >= 1 && !mbar_wait(smem_u32(tempty), (i - 1) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int s = 0; s < nk; ++s, ++q) {
                    const int st = q % S, sb = q % SB;
                    if (!mbar_wait(smem_u32(bfull + sb), (q / SB) & 1, limit, s_abort) ||
                        !mbar_wait(smem_u32(afull + st), (q / S) & 1, limit, s_abort)) {
                        set_abort(s_abort, P.status);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = tmem + kTmemA1 + (uint32_t)st * 64;   // gate A | up A (32 columns each)
                    const uint32_t bb = smem_u32(sB + sb * 16384);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t acc = (s | kk) != 0;
                        mma_f16_ts(tmem, a0 + kk * 8, desc_sw128(bb + kk * 32), idesc, acc);
                        mma_f16_ts(tmem + 128, a0 + 32 + kk * 8, desc_sw128(bb + kk * 32), idesc, acc);
                    }
                    mma_commit(smem_u32(aempty + st));
                    mma_commit(smem_u32(bempty + sb));
                }
                if (ok) mma_commit(smem_u32(tfull));
            }
            mma_commit(smem_u32(drain));   // every issued MMA completes before TMEM is freed
            mbar_wait(smem_u32(drain), 0, kDrainLimit, nullptr);
        }
    } else if (warp < kDequantWarps1) {
        // ------------------------------------------------ dequant
        // Warp w: matrix m = (w >> 2) & 1 (gate, up), rows 32 (w & 3) .. + 31 (the TMEM lanes
        // its position in a warpgroup allows), K-steps q of parity w >> 3.  Thread (m, r)
        // writes row r of matrix m's A stage in tensor memory: lane r, 32 columns of 16-bit
        // pairs in the codes' k order (x16 is stored in the same order).  The row's scales
        // and biases pass through a private double buffer of kScaleChunk1 groups: when a
        // chunk starts, the next one (of this tile or of the next tile) is requested with
        // cp.async, so the strided scale rows never stall the K loop.  The warps run
        // independently; each stops at the first failed wait.
        const int m = (warp >> 2) & 1, r = lane + 32 * (warp & 3), par = warp >> 3;
        const uint32_t a_lane = tmem + ((uint32_t)(r & ~31) << 16) + kTmemA1 + (uint32_t)m * 32;
        uint16_t *mysc = sScale + (size_t)tid * (4 * kScaleChunk1);   // [buffer][scale | bias][kScaleChunk1]
        const int nchunk = (G + kScaleChunk1 - 1) / kScaleChunk1;
        auto row_src = [&](const TileInfo &t, int c, const uint16_t *&ps, const uint16_t *&pb) -> size_t {
            ps = m == 0 ? (t.shared_e ? P.sgs : P.gs) : (t.shared_e ? P.sus : P.us);
            const size_t row = (size_t)(t.shared_e ? 0 : t.expert) * I + (size_t)(t.mb * 128 + r);
            if constexpr (BITS == kNvfp4) {            // 4 E4M3 bytes a group: groups 0-3 | 4-7 of the chunk
                pb = ps + 8;
                return row * (2 * G) + (size_t)c * 2 * kScaleChunk1;
            }
            pb = m == 0 ? (t.shared_e ? P.sgb : P.gb) : (t.shared_e ? P.sub : P.ub);
            return row * G + (size_t)c * kScaleChunk1;
        };
        auto fetch_chunk = [&](const TileInfo &t, int c, int buf) {     // one commit group per call
            if (t.mb * 128 + r < I) {
                const uint16_t *ps, *pb;
                const size_t off = row_src(t, c, ps, pb);
                uint16_t *d = mysc + buf * 2 * kScaleChunk1;
                cp_async16(smem_u32(d), ps + off);                     // 8 groups = 16 bytes
                cp_async16(smem_u32(d + kScaleChunk1), pb + off);
            }
            cp_async_commit();
        };
        auto load_chunk = [&](const TileInfo &t, int c, int buf) {      // the same with plain loads
            const bool row_ok = t.mb * 128 + r < I;
            const uint16_t *ps, *pb;
            const size_t off = row_src(t, c, ps, pb);
            uint16_t v[2][kScaleChunk1];
#pragma unroll
            for (int g = 0; g < kScaleChunk1; ++g) {
                // NVFP4: 16-bit slot g of a half holds bytes of group (4 half + g / 2) of the chunk
                const bool in0 = row_ok && c * kScaleChunk1 + (BITS == kNvfp4 ? g / 2 : g) < G;
                const bool in1 = row_ok && c * kScaleChunk1 + (BITS == kNvfp4 ? 4 + g / 2 : g) < G;
                v[0][g] = in0 ? ps[off + g] : (uint16_t)0;
                v[1][g] = in1 ? pb[off + g] : (uint16_t)0;
            }
            uint16_t *d = mysc + buf * 2 * kScaleChunk1;
#pragma unroll
            for (int g = 0; g < kScaleChunk1; ++g) {
                d[g] = v[0][g];
                d[kScaleChunk1 + g] = v[1][g];
            }
        };
        int q0 = 0, j = 0;                                 // q0: first K-step of the tile; j: chunks started
        bool ok = true;
        if (P.async_scales) fetch_chunk(tile_info(P.work, P.offsets, blockIdx.x, MB, P.E, Tk), 0, 0);
        for (int tau = blockIdx.x; tau < ntiles && ok; tau += gridDim.x, q0 += nk) {
            const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
            for (int c = 0; c < nchunk && ok; ++c) {
                if (P.async_scales) {
                    if (c + 1 < nchunk) fetch_chunk(ti, c + 1, (j + 1) & 1);
                    else if (tau + (int)gridDim.x < ntiles)
                        fetch_chunk(tile_info(P.work, P.offsets, tau + gridDim.x, MB, P.E, Tk), 0, (j + 1) & 1);
                    else cp_async_commit();
                    cp_async_wait_group<1>();                     // chunk j has landed
                } else {
                    load_chunk(ti, c, j & 1);
                }
                const uint16_t *cur = mysc + (j & 1) * 2 * kScaleChunk1;
                ++j;
                const uint4 sreg = *reinterpret_cast<const uint4 *>(cur);   // 8 groups (bf16 pairs)
                const uint4 breg = *reinterpret_cast<const uint4 *>(cur + kScaleChunk1);
                const int s_end = min(nk, (c + 1) * kScaleChunk1);
                for (int s = c * kScaleChunk1 + ((q0 + c * kScaleChunk1 + par) & 1); s < s_end; s += 2) {
                    const int q = q0 + s, st = q % S;
                    // the A stage of step q is free once the MMAs of step q - S are done; the
                    // fence orders this thread's tcgen05.st after those MMAs' reads
                    bool w_ok = q < S || mbar_wait(smem_u32(aempty + st), (q / S - 1) & 1, limit, s_abort);
                    tc_fence_after();
                    const int cs = q % CS;
                    w_ok = w_ok && mbar_wait(smem_u32(cfull + cs), (q / CS) & 1, limit, s_abort);
                    const int gi = s & 7;
                    const uint32_t sw = gi < 4 ? (gi < 2 ? sreg.x : sreg.y) : (gi < 6 ? sreg.z : sreg.w);
                    const uint32_t bw = gi < 4 ? (gi < 2 ? breg.x : breg.y) : (gi < 6 ? breg.z : breg.w);
                    __half2 sc, sc16, bc;
                    uint32_t nvs[2];                   // NVFP4: block scales 0,1 | 2,3 of the group (fp16x2)
                    if constexpr (BITS == kNvfp4) {
                        const uint32_t w4 = gi < 4 ? (gi < 2 ? (gi == 0 ? sreg.x : sreg.y) : (gi == 2 ? sreg.z : sreg.w))
                                                   : (gi < 6 ? (gi == 4 ? breg.x : breg.y) : (gi == 6 ? breg.z : breg.w));
                        nvs[0] = nv_e4m3x2_f16(w4);
                        nvs[1] = nv_e4m3x2_f16(w4 >> 16);
                    } else {
                        sc = bf16_to_h2((uint16_t)(gi & 1 ? sw >> 16 : sw));
                        sc16 = __hmul2(sc, __float2half2_rn(0.0625f));
                        bc = bf16_to_h2((uint16_t)(gi & 1 ? bw >> 16 : bw));
                    }
                    const uint8_t *cbase = sC + cs * CST + m * (CST / 2);
                    // tcgen05.st / wait::st are warp-collective: the lanes left the polling loops
                    // above at different iterations, so reconverge first
                    __syncwarp();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {           // inputs 32 hh .. 32 hh + 31
                        uint32_t av[16];
                        if (w_ok) {
                            uint32_t cw[cbits(BITS)];          // the 32 inputs' codes
                            if constexpr (BITS == 8) {
                                const uint4 w0 = *reinterpret_cast<const uint4 *>(cbase + swz64(r, 2 * hh));
                                const uint4 w1 = *reinterpret_cast<const uint4 *>(cbase + swz64(r, 2 * hh + 1));
                                cw[0] = w0.x, cw[1] = w0.y, cw[2] = w0.z, cw[3] = w0.w;
                                cw[4] = w1.x, cw[5] = w1.y, cw[6] = w1.z, cw[7] = w1.w;
                            } else {
                                const uint4 w = *reinterpret_cast<const uint4 *>(cbase + r * CB + hh * 16);
                                cw[0] = w.x, cw[1] = w.y, cw[2] = w.z, cw[3] = w.w;
                            }
#pragma unroll
                            for (int cc = 0; cc < 4; ++cc) {
                                uint4 d;
                                if constexpr (BITS == 8) d = dequant8_b8(cw[2 * cc], cw[2 * cc + 1], sc, bc);
                                else if constexpr (BITS == kNvfp4) d = nv_dequant8(cw[cc], nv_bcast(nvs[hh], cc >= 2));
                                else d = dequant8(cw[cc], sc, sc16, bc);
                                av[4 * cc] = d.x;
                                av[4 * cc + 1] = d.y;
                                av[4 * cc + 2] = d.z;
                                av[4 * cc + 3] = d.w;
                            }
                        } else {
#pragma unroll
                            for (int cc = 0; cc < 16; ++cc) av[cc] = 0u;
                        }
                        tmem_st16(a_lane + (uint32_t)st * 64 + (uint32_t)hh * 16, av);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    // One arrive per warp, after the warp has synchronised: with an arrive per
                    // thread, the MMAs were seen to read a stage before the stores of the last
                    // warps to arrive had landed.  A failed wait stops the whole warp.
                    if (__any_sync(0xffffffffu, !w_ok)) {
                        set_abort(s_abort, P.status);
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        tc_fence_before();
                        mbar_arrive(smem_u32(cempty + cs));    // the warp's code words are consumed
                        mbar_arrive(smem_u32(afull + st));
                    }
                }
            }
            if (*s_abort) break;
        }
        cp_async_wait_all();                               // no copy into shared memory outlives the CTA
    } else {
        // ------------------------------------------------ epilogue: h' = g' u' sigmoid(g' 2^e)
        // The accumulators hold g' = g 2^-e and u' = u 2^-e of token n (x' = x 2^-e); the stored fp16
        // h' = h 2^-2e stays inside the fp16 range whatever the size of x.  kEpiWarps1 warps: warp w
        // reads TMEM lanes 32 (w & 3) .. + 31 (the lanes its position in a warpgroup allows) and every
        // (kEpiWarps1 / 4)-th 16-column chunk of the accumulators, starting at chunk `half`.
        constexpr int kHalves = kEpiWarps1 / 4;
        const int quad = warp & 3, half = (warp - kWarpEpi1) >> 2, et = tid - kWarpEpi1 * 32;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        int i = 0;
        for (int tau = blockIdx.x; tau < ntiles; tau += gridDim.x, ++i) {
            const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
            const int N = (ti.ntok + 15) & ~15;
            // e and slot of each column (token n of the tile; 128 epilogue threads, 128 columns at
            // most), two tile buffers: the barrier of tile i + 1 orders every read of tile i before
            // tile i + 2 refills the buffer
            int *ce = s_col + (i & 1) * 256, *cf = ce + 128;
            for (int n = et; n < 128; n += 32 * kEpiWarps1) {
                int e = 0, f = -1;
                if (n < ti.ntok) {
                    int t = -1;
                    if (ti.shared_e) {
                        t = ti.tok0 + n;
                        f = Tk + t;
                    } else {
                        const int pos = ti.pbase + n;
                        f = (pos >= 0 && pos < Tk) ? __ldg(P.perm + pos) : -1;
                        if (f >= 0 && f < Tk) t = f / P.k;
                        else f = -1;
                    }
                    if (t >= 0) e = __ldg(P.xe + t);
                }
                ce[n] = e;
                cf[n] = f;
            }
            if (bar_any(3, 32 * kEpiWarps1, *s_abort)) break;
            bool got = mbar_wait(smem_u32(tfull), i & 1, limit, s_abort);
            got = __all_sync(0xffffffffu, got);              // tcgen05.ld needs the whole warp
            if (!got) set_abort(s_abort, P.status);
            if (bar_any(3, 32 * kEpiWarps1, !got)) break;    // the epilogue warps stop together
            tc_fence_after();
            const int erow = ti.mb * 128 + quad * 32 + lane;
            const int hcol = kperm_pos(erow);
            const uint32_t d0 = tmem + lane_base;
            float fg = 1.f, fu = 1.f;                     // NVFP4: the matrices' scales
            if constexpr (BITS == kNvfp4) {
                fg = __ldg(ti.shared_e ? P.sggs : P.ggs + ti.expert);
                fu = __ldg(ti.shared_e ? P.sugs : P.ugs + ti.expert);
            }
            if (16 * half >= N) {                             // no chunk of this parity: nothing to read
                tc_fence_before();
                mbar_arrive(smem_u32(tempty));
            }
            for (int n0 = 16 * half; n0 < N; n0 += 16 * kHalves) {
                uint32_t gv[16], uv[16];
                tmem_ld16(d0 + n0, gv);
                tmem_ld16(d0 + 128 + n0, uv);
                tmem_ld_wait();
                if (n0 + 16 * kHalves >= N) {             // this warp's last chunk: the MMAs may overwrite
                    tc_fence_before();
                    mbar_arrive(smem_u32(tempty));
                }
                if (erow < I) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = n0 + j;
                        if (n < ti.ntok) {
                            const float g = __uint_as_float(gv[j]) * fg, u = __uint_as_float(uv[j]) * fu;
                            const int e = ce[n];
                            const __half hq = __float2half_rn(__fdividef(g * u, 1.f + __expf(-g * pow2f(e))));
                            P.hs[(size_t)(ti.pbase + n) * I + hcol] = __half_as_ushort(hq);
                            if (P.h_out != nullptr && cf[n] >= 0) {
                                const float up = pow2f(e);
                                P.h_out[(size_t)cf[n] * I + erow] = __half2float(hq) * up * up;
                            }
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    pdl_wait();
}

// --------------------------------------------------------------- down GEMM
//
// Same structure; the token operand is the h tile of the expert's rows, loaded
// with TMA by a second thread of warp 4 as soon as each stage is free, and the
// epilogue adds p * y into the fp32 layer accumulator.
template <int S, int SB, int CS, int BITS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_down_kernel(const __grid_constant__ CUtensorMap map_dc, const __grid_constant__ CUtensorMap map_sdc,
                     const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_y,
                     const G2Params P)
{
    const int H = P.H, I = P.I, GI = I / kGroup, nk = GI, MB = (H + 127) / 128, Tk = P.T * P.k;
    constexpr int CB = code_row_bytes(BITS), CST = code_stage2(BITS);
    const size_t crow = (size_t)I * cbits(BITS) / 8;     // bytes of one weight row's codes
    const int ntiles = __ldg(P.nwork + 4) * MB;          // the big items lead the list
    // may start while the small-tile down GEMM still runs; waits for it before exiting
    if ((int)blockIdx.x >= ntiles) {
        pdl_wait();
        return;
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);
    uint8_t *sA = smem;                           // S x 16 KB
    uint8_t *sB = sA + S * 16384;                 // SB x 32 KB (256 rows x 128 B)
    uint8_t *sC = sB + SB * 32768;                // CS x CST
    uint16_t *sScale = reinterpret_cast<uint16_t *>(sC + CS * CST);    // [dequant thread][2][2][kScaleChunk1]
    float *sRed = reinterpret_cast<float *>(sScale + kDequantThreads * 4 * kScaleChunk1);   // [team][kRedBufs][kRedCols][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sRed + kEpiTeams2 * kRedBufs * kRedCols * 128);
    uint64_t *cfull = bars, *cempty = cfull + CS, *afull = cempty + CS, *aempty = afull + S;
    uint64_t *bfull = aempty + S, *bempty = bfull + SB;
    uint64_t *tfull = bempty + SB, *tempty = tfull + 2, *drain = tempty + 2;
    float *s_w = reinterpret_cast<float *>(drain + 1);          // [2][256]
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(s_w + 512);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(s_tmem), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < CS; ++s) {
            mbar_init(smem_u32(cfull + s), 1);
            mbar_init(smem_u32(cempty + s), kDequantThreads);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(afull + s), kDequantThreads);
            mbar_init(smem_u32(aempty + s), 1);
        }
        for (int s = 0; s < SB; ++s) {
            mbar_init(smem_u32(bfull + s), 1);
            mbar_init(smem_u32(bempty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(tfull + b), 1);
            mbar_init(smem_u32(tempty + b), 128 * kEpiTeams2);
        }
        mbar_init(smem_u32(drain), 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long limit = P.wait_limit;

    if (warp == kWarpTma) {
        if (lane == 0) {
            prefetch_map(&map_dc);
            prefetch_map(&map_sdc);
            // whole tiles (codes, scales, biases) requested from L2 in bulk one tile ahead
            auto prefetch_tile = [&](int tp) {
                if (tp >= ntiles) return;
                const TileInfo t2 = tile_info(P.work, P.offsets, tp, MB, P.E, Tk);
                const int rows = min(128, H - t2.mb * 128);
                const size_t wrow = (size_t)(t2.shared_e ? 0 : t2.expert * H) + t2.mb * 128;
                prefetch_rows((t2.shared_e ? P.sdc : P.dc) + wrow * crow, (uint32_t)(rows * crow));
                constexpr int kSb = BITS == kNvfp4 ? 4 : 2;
                const uint32_t sb = (uint32_t)rows * GI * kSb;
                prefetch_rows(reinterpret_cast<const uint8_t *>(t2.shared_e ? P.sds : P.ds) + wrow * GI * kSb, sb);
                if constexpr (BITS != kNvfp4) prefetch_rows((t2.shared_e ? P.sdb : P.db) + wrow * GI, sb);
            };
            prefetch_tile(blockIdx.x);
            int q = 0;
            bool ok = true;
            for (int tau = blockIdx.x; tau < ntiles && ok; tau += gridDim.x) {
                const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
                prefetch_tile(tau + gridDim.x);
                const CUtensorMap *md = ti.shared_e ? &map_sdc : &map_dc;
                const int wrow = (ti.shared_e ? 0 : ti.expert * H) + ti.mb * 128;
                for (int s = 0; s < nk; ++s, ++q) {
                    const int cs = q % CS;
                    if (q >= CS && !mbar_wait(smem_u32(cempty + cs), (q / CS - 1) & 1, limit, s_abort)) {
                        set_abort(s_abort, P.status);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(cfull + cs);
                    mbar_arrive_expect_tx(fb, CST);
                    tma_load_2d(smem_u32(sC + cs * CST), md, s * CB, wrow, fb);
                }
            }
            if (!ok || *s_abort)
                for (int d = (q > CS ? q - CS : 0); d < q; ++d)
                    mbar_wait(smem_u32(cfull + d % CS), (d / CS) & 1, kDrainLimit, nullptr);
        } else if (lane == 1) {
            // h tiles of the expert's rows (TMA), as soon as each stage is free
            prefetch_map(&map_h);
            int q = 0;
            bool ok = true;
            for (int tau = blockIdx.x; tau < ntiles && ok; tau += gridDim.x) {
                const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
                const int nbox = (((ti.ntok + 15) & ~15) + 31) / 32;
                for (int s = 0; s < nk; ++s, ++q) {
                    const int sb = q % SB;
                    if (q >= SB && !mbar_wait(smem_u32(bempty + sb), (q / SB - 1) & 1, limit, s_abort)) {
                        set_abort(s_abort, P.status);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(bfull + sb);
                    mbar_arrive_expect_tx(fb, (uint32_t)nbox * 4096);
                    for (int b = 0; b < nbox; ++b)
                        tma_load_2d(smem_u32(sB + sb * 32768 + b * 4096), &map_h, s * 64, ti.pbase + b * 32, fb);
                }
            }
            if (!ok || *s_abort)   // issued h tiles land before the CTA exits
                for (int d = (q > SB ? q - SB : 0); d < q; ++d)
                    mbar_wait(smem_u32(bfull + d % SB), (d / SB) & 1, kDrainLimit, nullptr);
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            int q = 0, i = 0;
            bool ok = true;
            for (int tau = blockIdx.x; tau < ntiles && ok; tau += gridDim.x, ++i) {
                const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
                const int N = (ti.ntok + 15) & ~15;
                const uint32_t idesc = idesc_f16_m128((uint32_t)N);
                const int buf = i & 1;
                if (i >= 2 && !mbar_wait(smem_u32(tempty + buf), ((i >> 1) - 1) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem + (uint32_t)buf * 256;
                for (int s = 0; s < nk; ++s, ++q) {
                    const int st = q % S, sb = q % SB;
                    if (!mbar_wait(smem_u32(bfull + sb), (q / SB) & 1, limit, s_abort) ||
                        !mbar_wait(smem_u32(afull + st), (q / S) & 1, limit, s_abort)) {
                        set_abort(s_abort, P.status);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t aa = smem_u32(sA + st * 16384), bb = smem_u32(sB + sb * 32768);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16(d0, desc_sw128(aa + kk * 32), desc_sw128(bb + kk * 32), idesc, (s | kk) != 0);
                    mma_commit(smem_u32(aempty + st));
                    mma_commit(smem_u32(bempty + sb));
                }
                if (ok) mma_commit(smem_u32(tfull + buf));
            }
            mma_commit(smem_u32(drain));
            mbar_wait(smem_u32(drain), 0, kDrainLimit, nullptr);
        }
    } else if (warp < 8) {
        // ------------------------------------------------ dequant: thread = half a row (4 chunks)
        // The row's scales and biases pass through a private double buffer of kScaleChunk1
        // groups, the next chunk (of this tile or of the next) requested with cp.async when
        // the current one starts: a tile has only I / 64 K-steps, so a synchronous load at
        // every tile start would stall the ring for a memory round trip each time.
        const int r = tid & 127, half = tid >> 7;
        uint16_t *mysc = sScale + (size_t)tid * (4 * kScaleChunk1);   // [buffer][scale | bias][kScaleChunk1]
        const int nchunk = (GI + kScaleChunk1 - 1) / kScaleChunk1;
        // NVFP4: 4 E4M3 bytes a group, groups 0-3 of a chunk in the scale half, 4-7 in the bias half
        constexpr int kCw = BITS == kNvfp4 ? 2 : 1;    // 16-bit words a group
        auto src_of = [&](const TileInfo &t, const uint16_t *&ps, const uint16_t *&pb) -> size_t {
            ps = t.shared_e ? P.sds : P.ds;
            pb = BITS == kNvfp4 ? ps + 8 : (t.shared_e ? P.sdb : P.db);
            return ((size_t)(t.shared_e ? 0 : t.expert) * H + (size_t)(t.mb * 128 + r)) * GI * kCw;
        };
        auto fetch_chunk = [&](const TileInfo &t, int c, int buf) {     // one commit group per call
            if (t.mb * 128 + r < H) {
                const uint16_t *ps, *pb;
                const size_t off = src_of(t, ps, pb) + (size_t)c * kScaleChunk1 * kCw;
                uint16_t *d = mysc + buf * 2 * kScaleChunk1;
                cp_async16(smem_u32(d), ps + off);
                cp_async16(smem_u32(d + kScaleChunk1), pb + off);
            }
            cp_async_commit();
        };
        auto load_chunk = [&](const TileInfo &t, int c, int buf) {      // the same with plain loads
            const bool row_ok = t.mb * 128 + r < H;
            const uint16_t *ps, *pb;
            const size_t off = src_of(t, ps, pb) + (size_t)c * kScaleChunk1 * kCw;
            uint16_t *d = mysc + buf * 2 * kScaleChunk1;
#pragma unroll
            for (int g = 0; g < kScaleChunk1; ++g) {
                const bool in0 = row_ok && c * kScaleChunk1 + (BITS == kNvfp4 ? g / 2 : g) < GI;
                const bool in1 = row_ok && c * kScaleChunk1 + (BITS == kNvfp4 ? 4 + g / 2 : g) < GI;
                d[g] = in0 ? ps[off + g] : (uint16_t)0;
                d[kScaleChunk1 + g] = in1 ? pb[off + g] : (uint16_t)0;
            }
        };
        int q = 0, j = 0;                                  // j: scale chunks started by this thread
        bool ok = true;
        if (P.async_scales) fetch_chunk(tile_info(P.work, P.offsets, blockIdx.x, MB, P.E, Tk), 0, 0);
        uint4 sreg = make_uint4(0, 0, 0, 0), breg = sreg;  // 8 groups' scales and biases (bf16 pairs)
        for (int tau = blockIdx.x; tau < ntiles; tau += gridDim.x) {
            const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
            for (int s = 0; s < nk && ok; ++s, ++q) {
                const int st = q % S;
                if (s % kScaleChunk1 == 0) {
                    const int c = s / kScaleChunk1;
                    if (P.async_scales) {
                        if (c + 1 < nchunk) fetch_chunk(ti, c + 1, (j + 1) & 1);
                        else if (tau + (int)gridDim.x < ntiles)
                            fetch_chunk(tile_info(P.work, P.offsets, tau + gridDim.x, MB, P.E, Tk), 0, (j + 1) & 1);
                        else cp_async_commit();
                        cp_async_wait_group<1>();                 // chunk j has landed
                    } else {
                        load_chunk(ti, c, j & 1);
                    }
                    const uint16_t *cur = mysc + (j & 1) * 2 * kScaleChunk1;
                    ++j;
                    sreg = *reinterpret_cast<const uint4 *>(cur);
                    breg = *reinterpret_cast<const uint4 *>(cur + kScaleChunk1);
                }
                if (q >= S && !mbar_wait(smem_u32(aempty + st), (q / S - 1) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                const int cs = q % CS;
                if (!mbar_wait(smem_u32(cfull + cs), (q / CS) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                const int gi = s & 7;
                const uint32_t sw = gi < 4 ? (gi < 2 ? sreg.x : sreg.y) : (gi < 6 ? sreg.z : sreg.w);
                const uint32_t bw = gi < 4 ? (gi < 2 ? breg.x : breg.y) : (gi < 6 ? breg.z : breg.w);
                uint8_t *aa = sA + st * 16384;
                if constexpr (BITS == kNvfp4) {            // inputs 32 half .. + 31: blocks 2 half, 2 half + 1
                    const uint32_t w4 = gi < 4 ? (gi < 2 ? (gi == 0 ? sreg.x : sreg.y) : (gi == 2 ? sreg.z : sreg.w))
                                               : (gi < 6 ? (gi == 4 ? breg.x : breg.y) : (gi == 6 ? breg.z : breg.w));
                    const uint32_t sb = nv_e4m3x2_f16(half ? w4 >> 16 : w4);
                    const uint4 w = *reinterpret_cast<const uint4 *>(sC + cs * CST + r * CB + half * 16);
                    const uint32_t cw[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(aa + swz128(r, half * 4 + c)) = nv_dequant8(cw[c], nv_bcast(sb, c >= 2));
                } else if constexpr (BITS == 8) {                 // inputs 32 half .. + 31: code chunks 2 half, 2 half + 1
                    const __half2 sd = bf16_to_h2((uint16_t)(gi & 1 ? sw >> 16 : sw));
                    const __half2 bd = bf16_to_h2((uint16_t)(gi & 1 ? bw >> 16 : bw));
                    const uint4 w0 = *reinterpret_cast<const uint4 *>(sC + cs * CST + swz64(r, 2 * half));
                    const uint4 w1 = *reinterpret_cast<const uint4 *>(sC + cs * CST + swz64(r, 2 * half + 1));
                    const uint32_t cw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(aa + swz128(r, half * 4 + c)) = dequant8_b8(cw[2 * c], cw[2 * c + 1], sd, bd);
                } else {
                    const __half2 sd = bf16_to_h2((uint16_t)(gi & 1 ? sw >> 16 : sw));
                    const __half2 sd16 = __hmul2(sd, __float2half2_rn(0.0625f));
                    const __half2 bd = bf16_to_h2((uint16_t)(gi & 1 ? bw >> 16 : bw));
                    const uint4 w = *reinterpret_cast<const uint4 *>(sC + cs * CST + r * CB + half * 16);
                    const uint32_t cw[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(aa + swz128(r, half * 4 + c)) = dequant8(cw[c], sd, sd16, bd);
                }
                mbar_arrive(smem_u32(cempty + cs));
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(afull + st));
            }
            if (bar_any(1, kDequantThreads, !ok || *s_abort)) break;   // the eight warps stop together
        }
        cp_async_wait_all();                               // no copy into shared memory outlives the CTA
    } else {
        // ------------------------------------------------ epilogue: the slot outputs 2^2e y
        // Team tm (warps 10 + 4 tm ..) takes chunks tm, tm + kEpiTeams2, ... of each tile with its own
        // chunk buffers and named barrier (id 2 + tm); barrier 5 spans both teams.
        constexpr int kEpiThreads = 128 * kEpiTeams2;
        const int quad = warp & 3, tm = (warp - kWarpEpi) >> 2, et = tid - kWarpEpi * 32, e = et & 127;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        float *const sRedT = sRed + tm * kRedBufs * kRedCols * 128;
        int i = 0, redc = 0;
        for (int tau = blockIdx.x; tau < ntiles; tau += gridDim.x, ++i) {
            const TileInfo ti = tile_info(P.work, P.offsets, tau, MB, P.E, Tk);
            const int N = (ti.ntok + 15) & ~15;
            const int buf = i & 1;
            float *wv = s_w + buf * 256;
            // factor 2^2e of each column (one per epilogue thread): the h tile holds h 2^-2e, the factor
            // undoes it (exact); NVFP4: times the matrix scale
            float fd = 1.f;
            if constexpr (BITS == kNvfp4) fd = __ldg(ti.shared_e ? P.sdgs : P.dgs + ti.expert);
            for (int n = et; n < 256; n += kEpiThreads) {
                float wgt = 0.f;
                if (n < ti.ntok) {
                    int t = -1;
                    if (ti.shared_e) {
                        t = ti.tok0 + n;
                    } else {
                        const int pos = ti.pbase + n;
                        const int f = (pos >= 0 && pos < Tk) ? __ldg(P.perm + pos) : -1;
                        if (f < 0 || f >= Tk) record_status(P.status, MOE_ERR_DEVICE);
                        else t = f / P.k;
                    }
                    if (t >= 0) {
                        const float up = pow2f(__ldg(P.xe + t));
                        wgt = up * up * fd;
                    }
                }
                wv[n] = wgt;
            }
            if (bar_any(5, kEpiThreads, *s_abort)) break;
            bool got = mbar_wait(smem_u32(tfull + buf), (i >> 1) & 1, limit, s_abort);
            got = __all_sync(0xffffffffu, got);              // tcgen05.ld needs the whole warp
            if (!got) set_abort(s_abort, P.status);
            if (bar_any(5, kEpiThreads, !got)) break;        // the epilogue warps stop together
            tc_fence_after();
            // 2^2e y of 16 columns at a time into a shared-memory chunk [column][row], then one tiled
            // store of the chunk: its columns are 16 consecutive rows of yslot (expert-sorted positions)
            // and the tile's 128 rows of H are contiguous there (a ragged last chunk: one bulk store per
            // column).  Every (slot, row) is written once; the slots are summed afterwards in a fixed
            // order.
            const int rloc = quad * 32 + lane, nrow = min(128, H - ti.mb * 128);
            const uint32_t d0 = tmem + lane_base + (uint32_t)buf * 256;
            if (tm * kRedCols >= N) {                     // no chunk for this team: nothing to read
                tc_fence_before();
                mbar_arrive(smem_u32(tempty + buf));
            }
            for (int n0 = tm * kRedCols; n0 < N; n0 += kEpiTeams2 * kRedCols, ++redc) {
                uint32_t v[16];
                tmem_ld16(d0 + n0, v);
                tmem_ld_wait();
                if (n0 + kEpiTeams2 * kRedCols >= N) {    // this team's last chunk read: the MMAs may overwrite
                    tc_fence_before();
                    mbar_arrive(smem_u32(tempty + buf));
                }
                float *red = sRedT + (redc % kRedBufs) * kRedCols * 128;
                if (e < kRedCols) bulk_wait_read<kRedBufs - 1>();   // this buffer's stores (kRedBufs chunks ago) have read it
                named_bar(2 + tm, 128);
#pragma unroll
                for (int j = 0; j < 16; ++j) red[j * 128 + rloc] = wv[n0 + j] * __uint_as_float(v[j]);
                fence_proxy_async_smem();
                named_bar(2 + tm, 128);
                if (e < kRedCols) {
                    if (n0 + kRedCols <= ti.ntok) {
                        if (e == 0) tma_store_2d(&map_y, ti.mb * 128, ti.pbase + n0, smem_u32(red));
                    } else if (n0 + e < ti.ntok) {
                        bulk_store(P.yslot + (size_t)(ti.pbase + n0 + e) * H + ti.mb * 128, smem_u32(red + e * 128),
                                   (uint32_t)nrow * 4);
                    }
                    bulk_commit();
                }
            }
            if (bar_any(5, kEpiThreads, *s_abort)) break;   // wv of this buffer is reused two tiles later
        }
        bulk_wait<0>();                                   // every bulk store has completed
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    pdl_wait();
}

// x (bf16) -> x' = x 2^-e per token (e from the row's largest |x|: max |x'| in [1, 2); exact) as
// fp16 in the codes' k order within each chunk of 8, e per token, and per token and group of 64
// the sum of the stored fp16 values (each chunk in element order, then a fixed shuffle tree over
// the group's eight chunks; the small-tile GEMM's bias term).  One warp per token: lane l takes the
// row's chunks l, l + 32, ...; a group's chunks sit in eight consecutive lanes.
__global__ void convert_x_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ x16, float *__restrict__ xsum,
                                 int *__restrict__ xe, int T, int H)
{
    const int lane = threadIdx.x & 31, cpr = H / 8, G = H / kGroup;
    const int wpb = blockDim.x >> 5, nw = gridDim.x * wpb;
    for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += nw) {
        const uint4 *xr = x + (size_t)t * cpr;
        uint32_t mx = 0;
        for (int c = lane; c < cpr; c += 32) {
            const uint4 v = xr[c];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        const int e = row_scale_exponent(mx);
        const float sc = pow2f(-e);
        for (int c0 = 0; c0 < cpr; c0 += 32) {          // every lane runs every round (the shuffles)
            const int c = c0 + lane;
            float sum = 0.f;
            if (c < cpr) {
                const uint4 v = xr[c];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                float f[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    f[2 * j] = __uint_as_float(w[j] << 16) * sc;
                    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u) * sc;
                }
                const __half2 h0 = __floats2half2_rn(f[0], f[4]), h1 = __floats2half2_rn(f[1], f[5]);
                const __half2 h2 = __floats2half2_rn(f[2], f[6]), h3 = __floats2half2_rn(f[3], f[7]);
                uint4 o;
                o.x = h2u(h0);
                o.y = h2u(h1);
                o.z = h2u(h2);
                o.w = h2u(h3);
                x16[(size_t)t * cpr + c] = o;
                const __half2 hs[4] = {h0, h1, h2, h3};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    sum += __low2float(hs[j]);
                    sum += __high2float(hs[j]);
                }
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            if (c < cpr && (c & 7) == 0) xsum[(size_t)t * G + (c >> 3)] = sum;
        }
        if (lane == 0) xe[t] = e;
    }
}

// ------------------------------------------------------------------ host side

size_t g1_smem(int cs, int bits)
{
    return 1024 + kStagesB1 * 16384 + (size_t)cs * code_stage1(bits) + kDequantWarps1 * 32 * 4 * kScaleChunk1 * 2 +
           2 * 256 * 4 + 8 * (2 * cs + 2 * kStagesA1 + 2 * kStagesB1 + 5) + 256 * 4 + 16;
}
size_t g2_smem(int cs, int bits)
{
    return 1024 + kStagesA2 * 16384 + kStagesB2 * 32768 + (size_t)cs * code_stage2(bits) +
           kDequantThreads * 4 * kScaleChunk1 * 2 + kEpiTeams2 * kRedBufs * kRedCols * 128 * 4 +
           8 * (2 * cs + 2 * kStagesA2 + 2 * kStagesB2 + 5) + 512 * 4 + 16;
}

// Launch allowed (pdl) to begin while the previous kernel of the stream still runs.
template <typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kern)(Args...), int grid, int threads, size_t smem, cudaStream_t st,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}


}  // namespace

cudaError_t launch_prefill_experts(const PrefillArgs &a, cudaStream_t st)
{
    const int H = a.H, I = a.I, E = a.E, T = a.T, k = a.k;
    // x -> x' = x 2^-e per token, fp16, K-permuted (one warp per token)
    {
        const unsigned grid = (unsigned)std::min<int>((T + 7) / 8, 152 * 8);
        convert_x_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4 *>(a.x), reinterpret_cast<uint4 *>(a.x16),
                                               a.xsum, a.xe, T, H);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaSuccess;

    if (a.bits != 4 && a.bits != 8 && a.bits != kNvfp4) return cudaErrorInvalidValue;
    const bool b8 = a.bits == 8, nv = a.bits == kNvfp4;
    CUtensorMap mgc, muc, msgc, msuc, mdc, msdc, mh, my;
    const CUtensorMapSwizzle sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
    // code boxes: 32 bytes (4-bit, unswizzled) or 64 bytes with the 64-byte swizzle (8-bit) of 128 rows
    const CUtensorMapSwizzle csw = b8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE;
    const uint32_t cbox = (uint32_t)code_row_bytes(a.bits);
    const uint64_t hrow = (uint64_t)H * cbits(a.bits) / 8, irow = (uint64_t)I * cbits(a.bits) / 8;   // code bytes per row
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int ns = a.has_shared ? 1 : 0;
    bool ok = make_map_2d(&mgc, a.gate.codes, u8, 1, hrow, (uint64_t)E * I, cbox, 128, csw) &&
              make_map_2d(&muc, a.up.codes, u8, 1, hrow, (uint64_t)E * I, cbox, 128, csw) &&
              make_map_2d(&mdc, a.down.codes, u8, 1, irow, (uint64_t)E * H, cbox, 128, csw) &&
              make_map_2d(&mh, a.hs, f16, 2, I, (uint64_t)T * k + (uint64_t)T, 64, 32, sw128) &&
              make_map_2d(&my, a.yslot, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, (uint64_t)T * k + (uint64_t)T, 128,
                          kRedCols, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (ns)
        ok = ok && make_map_2d(&msgc, a.s_gate.codes, u8, 1, hrow, I, cbox, 128, csw) &&
             make_map_2d(&msuc, a.s_up.codes, u8, 1, hrow, I, cbox, 128, csw) &&
             make_map_2d(&msdc, a.s_down.codes, u8, 1, irow, H, cbox, 128, csw);
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
    p1.xe = a.xe;
    p1.h_out = a.h_out;
    p1.gc = a.gate.codes;
    p1.uc = a.up.codes;
    p1.sgc = a.has_shared ? a.s_gate.codes : a.gate.codes;
    p1.suc = a.has_shared ? a.s_up.codes : a.up.codes;
    p1.gs = a.gate.scales;
    p1.gb = a.gate.biases;
    p1.us = a.up.scales;
    p1.ub = a.up.biases;
    p1.sgs = a.s_gate.scales;
    p1.sgb = a.s_gate.biases;
    p1.sus = a.s_up.scales;
    p1.sub = a.s_up.biases;
    p1.ggs = a.gate.gscale;
    p1.ugs = a.up.gscale;
    p1.sggs = a.has_shared ? a.s_gate.gscale : a.gate.gscale;
    p1.sugs = a.has_shared ? a.s_up.gscale : a.up.gscale;
    p1.status = a.status;
    p1.T = T;
    p1.H = H;
    p1.I = I;
    p1.E = E;
    p1.k = k;
    {
        const uint16_t *sc[8] = {p1.gs, p1.gb, p1.us, p1.ub, p1.sgs, p1.sgb, p1.sus, p1.sub};
        bool al = (H / kGroup) % 8 == 0;
        for (const uint16_t *ptr : sc) al = al && (ptr == nullptr || reinterpret_cast<uintptr_t>(ptr) % 16 == 0);
        p1.async_scales = al ? 1 : 0;
    }
    p1.wait_limit = a.wait_limit;
    const size_t s1 = b8 ? g1_smem(kCodeStages1B8, 8) : g1_smem(kCodeStages1, 4);
    auto k1 = b8 ? gemm_gateup_kernel<kStagesA1, kStagesB1, kCodeStages1B8, 8>
                 : nv ? gemm_gateup_kernel<kStagesA1, kStagesB1, kCodeStages1, kNvfp4>
                      : gemm_gateup_kernel<kStagesA1, kStagesB1, kCodeStages1, 4>;
    cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
    const int tiles1 = a.max_w1 * ((I + 127) / 128);
    const bool small = prefill_small_fits(H, I, a.bits);   // items of small experts: mma.sync tiles (nwork[3] on)
    if (small && (e = launch_small_gateup(a, st)) != cudaSuccess) return e;
    // behind the small-tile kernel (if any) as its programmatic dependent
    if ((e = launch_pdl(small, k1, std::min(device_sm_count(), tiles1), kThreads1, s1, st, mgc, muc, msgc, msuc, p1)) !=
        cudaSuccess)
        return e;

    G2Params p2{};
    p2.nwork = a.nwork;
    p2.work = a.work_g2;
    p2.offsets = a.offsets;
    p2.perm = a.perm;
    p2.xe = a.xe;
    p2.yslot = a.yslot;
    p2.dc = a.down.codes;
    p2.sdc = a.has_shared ? a.s_down.codes : a.down.codes;
    p2.ds = a.down.scales;
    p2.db = a.down.biases;
    p2.sds = a.s_down.scales;
    p2.sdb = a.s_down.biases;
    p2.dgs = a.down.gscale;
    p2.sdgs = a.has_shared ? a.s_down.gscale : a.down.gscale;
    p2.status = a.status;
    p2.T = T;
    p2.H = H;
    p2.I = I;
    p2.E = E;
    p2.k = k;
    {
        const uint16_t *sc[4] = {p2.ds, p2.db, p2.sds, p2.sdb};
        bool al = (I / kGroup) % 8 == 0;
        for (const uint16_t *ptr : sc) al = al && (ptr == nullptr || reinterpret_cast<uintptr_t>(ptr) % 16 == 0);
        p2.async_scales = al ? 1 : 0;
    }
    p2.wait_limit = a.wait_limit;
    const size_t s2 = b8 ? g2_smem(kCodeStages2B8, 8) : g2_smem(kCodeStages2, 4);
    auto k2 = b8 ? gemm_down_kernel<kStagesA2, kStagesB2, kCodeStages2B8, 8>
                 : nv ? gemm_down_kernel<kStagesA2, kStagesB2, kCodeStages2, kNvfp4>
                      : gemm_down_kernel<kStagesA2, kStagesB2, kCodeStages2, 4>;
    cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
    const int tiles2 = a.max_w2 * ((H + 127) / 128);
    if (small && (e = launch_small_down(a, st)) != cudaSuccess) return e;
    return launch_pdl(small, k2, std::min(device_sm_count(), tiles2), kThreads, s2, st, mdc, msdc, mh, my, p2);
}

}  // namespace qmoe
