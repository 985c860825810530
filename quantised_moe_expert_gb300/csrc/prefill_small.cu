// Small-tile grouped expert GEMMs of the prefill path: the experts of at most kSmallN
// tokens, one work item each (at T = 512 over 256 experts that is every routed expert,
// ~16 tokens each).  They run first; the tensor-memory GEMMs of the larger experts are
// launched behind them as programmatic dependents and fill the SMs these kernels free.
//
// At that size each int4 weight meets only a few tokens, so the GEMMs stream weights:
// the prefill pages' point that both stacks became weight-bandwidth bound (page "POC for
// qwen3.5 / qwen3.6 support optimized for AGX Orin", Phase 1-4) holds here too.  A
// tcgen05 MMA with M = 128, K = 16 costs ~46 cycles for any N <= 64 on this GPU, and the
// dequantisation of every weight to fp16 comes on top; so these tiles use the decode
// GEMV's arithmetic on mma.sync instead, with the codes used exactly:
//     sum_j w_j x_j = s * sum_j (q_j - 8) x_j + (b + 8 s) * sum_j x_j
// over each group of 64 inputs, q - 8 exact in fp16 (nib8_signed), fp32 accumulation, scale
// and bias per group in fp32.  The tensor-memory kernels keep the experts with many tokens.
//
// Gate/up kernel (one CTA per SM, persistent over tiles = item x 128-row block of I):
//   warp 16 (one thread) streams each K-step's gate and up code boxes (128 rows x 32
//   bytes) with TMA through a ring, and each tile's scale and bias rows with bulk copies
//   into a double buffer; warps 17-18 take the K-steps in turn and gather the item's token
//   rows of x16 (fp16, the codes' k order) into 128-byte-swizzled stages with cp.async
//   (warp 17 also the tile's group sums of x); warp w < 16 owns rows 16 (w % 8) .. + 15 of
//   matrix w / 8 (gate, up) for all the item's tokens.  At the end of a tile the up warps
//   hand their sums to the gate warps through shared memory, which store h = silu(g) * u
//   as fp16 in the codes' k order.
// Down kernel (tiles of 256 rows of H): the same with the down codes, the item's h rows
//   (TMA, the same swizzle) and the group sums of h that the gate/up kernel's epilogue
//   stored; warp w < 16 owns rows 16 w .. + 15; the epilogue writes each slot's expert
//   output y_e (fp32) once into the slot buffer.
#include <algorithm>

#include "kernels.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace qmoe {
namespace {

using namespace tc;

constexpr int kSCodeStages = 8;     // down: 4 KB h + 2 x 4 KB codes per stage (one K-step)
constexpr int kSCompute = 16;       // compute warps of both kernels
constexpr int kSWarpTma = 16, kSWarpAux = 17;
constexpr int kSThreads1 = 32 * (kSCompute + 1);           // gate/up: + the producer warp (544)
constexpr int kSThreads2 = 32 * (kSWarpAux + 1);           // down: + the column helper warp (576)
// Gate/up stages cover four K-steps: the code boxes are then 128 bytes wide (whole lines of
// each row, stored with the 128-byte swizzle), and each token row's 4 x 64 inputs one bulk copy.
constexpr int kG1Steps = 4, kG1Stages = 2;
constexpr int kG1XRow = 4 * 128 + 16;                       // x row stride: 8 rows on distinct banks
constexpr int kG1Stage = (2 * 16384 + kSmallN * kG1XRow + 1023) / 1024 * 1024;   // gate | up codes | x rows
constexpr long long kSDrainLimit = 1ll << 22;
static_assert(kSmallN == 32, "one loader lane per token row, four n8 tiles");
static_assert(kG1Stage % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled code boxes");

// Named barrier over the compute warps that also ORs a predicate (a uniform stop decision).  The
// non-aligned form, each warp brought back together first: lanes may arrive apart.
__device__ __forceinline__ bool compute_any(bool pred)
{
    __syncwarp();
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(kSCompute * 32)
        : "memory");
    return r != 0;
}

struct SmallParams {
    const int32_t *nwork;
    const WorkItem *work;
    const int32_t *offsets;
    const int32_t *perm;
    uint16_t *hs;                      // fp16 [T*k + T, I] (k order), expert-sorted rows: h' = h 2^-2e
    const uint16_t *x16;               // fp16 [T, H] (k order): x' = x 2^-e
    const float *xsum;                 // f32 [T, H / 64]
    const int *xe;                     // i32 [T]: e of each token
    float *h_out;                      // f32 [T*k + T, I] h per slot (stage output), or null
    float *yslot;                      // f32 [T*k + T, H] each slot's expert output before its pick weight, rows in
                                       // expert-sorted position order (the rows of the h tiles)
    float *hsum;                       // f32 [T*k + T, I / 64]: group sums of the stored (fp16) h
    const uint8_t *c0, *c1, *sc0, *sc1;            // codes (routed, shared) for L2 prefetch: gate, up / down
    const uint16_t *s0, *b0, *s1, *b1;             // routed scales, biases: gate, up / down
    const uint16_t *ss0, *sb0, *ss1, *sb1;         // shared expert
    int *status;
    int T, H, I, E, k;
    long long wait_limit;
    DequantK dq;                       // code conversion constants (kDequantK)
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk)
{
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void mma16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int kperm_pos(int i) { return (i & ~7) | ((i & 3) << 1) | ((i >> 2) & 1); }

// Scale rows in shared memory are read 4 groups at a time into registers (one 8-byte load
// when the row length allows it): per-step 2-byte loads of 8 different rows would hit the
// same banks.
__device__ __forceinline__ uint2 scale_window(const uint16_t *base, int row, int len, int s4)
{
    if ((len & 3) == 0) return *reinterpret_cast<const uint2 *>(base + row * len + s4);
    uint32_t v[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const uint32_t lo = s4 + 2 * e < len ? base[row * len + s4 + 2 * e] : 0u;
        const uint32_t hi = s4 + 2 * e + 1 < len ? base[row * len + s4 + 2 * e + 1] : 0u;
        v[e] = lo | (hi << 16);
    }
    return make_uint2(v[0], v[1]);
}
__device__ __forceinline__ float scale_pick(const uint2 &w, int e)
{
    const uint32_t x = e < 2 ? w.x : w.y;
    return bf16_bits_to_float((uint16_t)((e & 1) ? x >> 16 : x));
}

__device__ __forceinline__ void set_abort(volatile int *abort, int *status)
{
    *abort = 1;
    record_status(status, MOE_ERR_TIMEOUT);
}

struct STile {
    int expert, tok0, ntok, mb, pbase;
    bool shared_e;
};

// Tile tau: small item nbig + tau / MB, 128-row block tau % MB.
__device__ __forceinline__ STile stile(const SmallParams &P, int nbig, int tau, int MB, int Tk)
{
    const WorkItem it = P.work[nbig + tau / MB];
    STile t;
    t.expert = it.expert;
    t.tok0 = it.tok0;
    t.ntok = it.ntok;
    t.mb = tau % MB;
    t.shared_e = it.expert == P.E;
    t.pbase = t.shared_e ? Tk + it.tok0 : __ldg(P.offsets + it.expert) + it.tok0;
    return t;
}

// The producer's lanes wait together (one poll, the answer broadcast).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, long long limit, volatile int *abort)
{
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, limit, abort);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// ------------------------------------------------------------------ gate/up
__global__ void __launch_bounds__(kSThreads1, 1)
    small_gateup_kernel(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_u,
                        const __grid_constant__ CUtensorMap map_sg, const __grid_constant__ CUtensorMap map_su,
                        const SmallParams P)
{
    pdl_trigger();   // the tensor-memory gate/up GEMM may take every SM this grid frees
    const int H = P.H, I = P.I, G = H / kGroup, nk = G, MB = (I + 127) / 128, Tk = P.T * P.k;
    const int nst = nk / kG1Steps;                  // stages per tile (H % 256 == 0)
    const int nbig = __ldg(P.nwork + 3);
    const int ntiles = (__ldg(P.nwork + 1) - nbig) * MB;
    if ((int)blockIdx.x >= ntiles) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);
    uint8_t *sR = smem;                                                    // kG1Stages x kG1Stage
    float *sU = reinterpret_cast<float *>(sR + kG1Stages * kG1Stage);      // [2][8 warps][32 lanes][16]: up sums
    uint16_t *sS = reinterpret_cast<uint16_t *>(sU + 2 * 8 * 32 * 16);     // [2][4][128][G]
    const int XS = G + 4;                  // group-sum row stride: distinct banks for the columns a warp reads
    float *sX = reinterpret_cast<float *>(sS + 2 * 4 * 128 * G);           // [2][kSmallN][XS]
    float *sH = sX + 2 * kSmallN * XS;                                     // [2][8 gate warps][32]: h sums
    int *s_e = reinterpret_cast<int *>(sH + 2 * 8 * 32);                   // [3][kSmallN]: e of each column
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_e + 3 * kSmallN);
    uint64_t *sfull = bars, *sempty = sfull + kG1Stages, *tfull = sempty + kG1Stages, *tempty = tfull + 2;
    volatile int *s_abort = reinterpret_cast<volatile int *>(tempty + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kG1Stages; ++s) {
            mbar_init(smem_u32(sfull + s), 1);
            mbar_init(smem_u32(sempty + s), kSCompute);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(tfull + b), 1);
            mbar_init(smem_u32(tempty + b), kSCompute);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const long long limit = P.wait_limit;
    const DequantK dq = P.dq;

    if (warp == kSCompute) {
        // ------------------------------------------------ producer: lane 0 the code boxes (TMA) and scale
        // rows, lane n token row n (its group sums per tile, its 256 inputs per stage; bulk copies)
        if (lane == 0) {
            prefetch_map(&map_g);
            prefetch_map(&map_u);
            prefetch_map(&map_sg);
            prefetch_map(&map_su);
        }
        // no L2 prefetch of the next tile: the code boxes are whole 128-byte lines, and lines
        // requested a tile ahead were partly evicted before use (~40% more DRAM reads)
        auto rows_of = [&](const STile &t) { return min(128, I - t.mb * 128); };
        int q = 0, i = 0;                           // q: stages issued
        bool ok = true;
        for (int tau = blockIdx.x; tau < ntiles && ok; tau += gridDim.x, ++i) {
            const STile t = stile(P, nbig, tau, MB, Tk);
            int row = -1;
            if (lane < t.ntok) {
                if (t.shared_e) {
                    row = t.tok0 + lane;
                } else {
                    const int pos = t.pbase + lane;
                    const int f = (pos >= 0 && pos < Tk) ? __ldg(P.perm + pos) : -1;
                    if (f < 0 || f >= Tk) record_status(P.status, MOE_ERR_DEVICE);
                    else row = f / P.k;
                }
            }
            const int nrows = __popc(__ballot_sync(0xffffffffu, row >= 0));
            const int buf = i & 1;
            if (i >= 2 && !warp_wait(smem_u32(tempty + buf), ((i >> 1) - 1) & 1, limit, s_abort)) {
                set_abort(s_abort, P.status);
                break;
            }
            const size_t wrow = (size_t)(t.shared_e ? 0 : t.expert * I) + t.mb * 128;
            const uint32_t sbytes = (uint32_t)rows_of(t) * G * 2;
            const uint32_t tb = smem_u32(tfull + buf);
            // e of column `lane` for the gate warps' epilogue, in tile slot i % 3: it is refilled (tile
            // i + 3) only after every compute warp released tile i + 1, i.e. after tile i's epilogue;
            // ordered before lane 0's arrival on the tile barrier by the warp barrier
            s_e[(i % 3) * kSmallN + lane] = row >= 0 ? __ldg(P.xe + row) : 0;
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(tb, 4 * sbytes + (uint32_t)nrows * G * 4);
                const uint16_t *src[4] = {t.shared_e ? P.ss0 : P.s0, t.shared_e ? P.sb0 : P.b0,
                                          t.shared_e ? P.ss1 : P.s1, t.shared_e ? P.sb1 : P.b1};
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    bulk_load(smem_u32(sS + (buf * 4 + a) * 128 * G), src[a] + wrow * G, sbytes, tb);
            }
            __syncwarp();
            if (row >= 0) bulk_load(smem_u32(sX + (buf * kSmallN + lane) * XS), P.xsum + (size_t)row * G, G * 4, tb);
            const uint16_t *src = row >= 0 ? P.x16 + (size_t)row * H : nullptr;
            const CUtensorMap *mg = t.shared_e ? &map_sg : &map_g;
            const CUtensorMap *mu = t.shared_e ? &map_su : &map_u;
#pragma unroll 1
            for (int k4 = 0; k4 < nst; ++k4, ++q) {
                const int st = q % kG1Stages;
                if (q >= kG1Stages &&
                    !warp_wait(smem_u32(sempty + st), (q / kG1Stages - 1) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                uint8_t *stg = sR + st * kG1Stage;
                const uint32_t fb = smem_u32(sfull + st);
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, 2 * 16384 + (uint32_t)nrows * 512);
                    tma_load_2d(smem_u32(stg), mg, k4 * 128, (int)wrow, fb);
                    tma_load_2d(smem_u32(stg + 16384), mu, k4 * 128, (int)wrow, fb);
                }
                __syncwarp();
                if (src) bulk_load(smem_u32(stg + 32768 + lane * kG1XRow), src + k4 * 256, 512, fb);
            }
        }
        // every issued copy lands before the CTA exits
        if (lane == 0) {
            for (int d = (q > kG1Stages ? q - kG1Stages : 0); d < q; ++d)
                mbar_wait(smem_u32(sfull + d % kG1Stages), (d / kG1Stages) & 1, kSDrainLimit, nullptr);
            for (int b = 0; b < 2 && b < i; ++b) {
                const int last = i - 1 - ((i - 1 - b) & 1);   // the last tile that used buffer (i - 1 - b) & 1
                mbar_wait(smem_u32(tfull + (last & 1)), (last >> 1) & 1, kSDrainLimit, nullptr);
            }
        }
        return;
    }

    // ---------------------------------------------------- compute warps: matrix w / 8, rows 16 (w % 8) ..
    const int g = lane >> 2, t4 = lane & 3, m = warp >> 3, rw = warp & 7;
    const int r0 = rw * 16 + g;                     // rows r0 and r0 + 8 of the tile
    // byte offsets, inside a stage's 128-byte-swizzled box, of row r0 and row r0 + 8 (row r of a
    // box sits at (r / 8) * 1024 + (r % 8) * 128 with its 16-byte chunk c at c ^ (r % 8); r0 % 8 = g)
    const uint32_t crow0 = m * 16384 + (uint32_t)(2 * rw) * 1024 + g * 128, crow1 = crow0 + 1024;
    int q = 0, i = 0;
    for (int tau = blockIdx.x; tau < ntiles; tau += gridDim.x, ++i) {
        const STile t = stile(P, nbig, tau, MB, Tk);
        const int buf = i & 1, ncol = t.ntok;
        bool w_ok = mbar_wait(smem_u32(tfull + buf), (i >> 1) & 1, limit, s_abort);
        const uint16_t *ssc = sS + (buf * 4 + 2 * m) * 128 * G;   // this matrix's scales, then biases
        const float *sxs = sX + buf * kSmallN * XS;
        float acc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
#pragma unroll 1
        for (int k4 = 0; k4 < nst && w_ok; ++k4, ++q) {
            const int st = q % kG1Stages;
            w_ok = mbar_wait(smem_u32(sfull + st), (q / kG1Stages) & 1, limit, s_abort);
            if (!w_ok) break;
            const uint8_t *stg = sR + st * kG1Stage;
            const uint2 ws0 = scale_window(ssc, r0, G, k4 * 4), ws1 = scale_window(ssc, r0 + 8, G, k4 * 4);
            const uint2 wb0 = scale_window(ssc + 128 * G, r0, G, k4 * 4);
            const uint2 wb1 = scale_window(ssc + 128 * G, r0 + 8, G, k4 * 4);
#pragma unroll
            for (int e = 0; e < kG1Steps; ++e) {
                const int s = k4 * 4 + e;
                // this lane's 8 code bytes of step e: 16-byte chunk 2 e + t4 / 2, half t4 % 2
                const uint32_t co = (((2 * e + (t4 >> 1)) ^ g) << 4) | ((t4 & 1) << 3);
                const uint2 c0 = *reinterpret_cast<const uint2 *>(stg + crow0 + co);
                const uint2 c1 = *reinterpret_cast<const uint2 *>(stg + crow1 + co);
                const float s0 = scale_pick(ws0, e), s1 = scale_pick(ws1, e);
                const float k0 = fmaf(8.f, s0, scale_pick(wb0, e));
                const float k1 = fmaf(8.f, s1, scale_pick(wb1, e));
                uint32_t aa[2][8];
                nib8_signed(c0.x, aa[0], dq);
                nib8_signed(c0.y, aa[0] + 4, dq);
                nib8_signed(c1.x, aa[1], dq);
                nib8_signed(c1.y, aa[1] + 4, dq);
                const uint8_t *xb = stg + 32768 + g * kG1XRow + e * 128 + t4 * 32;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j * 8 >= ncol) break;
                    // token column j * 8 + g; rows past ncol hold stale data, only their own columns see it
                    const uint4 lo = *reinterpret_cast<const uint4 *>(xb + j * 8 * kG1XRow);
                    const uint4 hi = *reinterpret_cast<const uint4 *>(xb + j * 8 * kG1XRow + 16);
                    const uint32_t bp[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm)
                        mma16816_f16(d, aa[0][2 * mm], aa[1][2 * mm], aa[0][2 * mm + 1], aa[1][2 * mm + 1], bp[2 * mm],
                                     bp[2 * mm + 1]);
                    const int cA = j * 8 + 2 * t4;
                    const float sxA = sxs[cA * XS + s], sxB = sxs[(cA + 1) * XS + s];
                    acc[j][0] = fmaf(s0, d[0], fmaf(k0, sxA, acc[j][0]));
                    acc[j][1] = fmaf(s0, d[1], fmaf(k0, sxB, acc[j][1]));
                    acc[j][2] = fmaf(s1, d[2], fmaf(k1, sxA, acc[j][2]));
                    acc[j][3] = fmaf(s1, d[3], fmaf(k1, sxB, acc[j][3]));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(sempty + st));
        }
        if (!w_ok) set_abort(s_abort, P.status);
        __syncwarp();
        if (lane == 0 && w_ok) mbar_arrive(smem_u32(tempty + buf));   // scales and group sums no longer read
        // the up warps hand their sums to the gate warps of the same rows (buffer by tile parity)
        float *xu = sU + ((buf * 8 + rw) * 32 + lane) * 16;
        if (m == 1)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) xu[j * 4 + e] = acc[j][e];
        if (compute_any(!w_ok)) {                   // all sixteen warps stop together
            set_abort(s_abort, P.status);
            break;
        }
        if (m == 0) {
            // h' = g' u' sigmoid(g' 2^e) for the tile's rows and tokens (g' = g 2^-e, u' = u 2^-e: x is
            // pre-scaled per token; h' = h 2^-2e), fp16, at the row's k-order column; and per token the
            // sum of the stored h' over each group of 64 rows (the down GEMM's bias term): this warp's
            // 16 rows by shuffles, the group's four warps through shared memory in order
            float *hp = sH + (buf * 8 + rw) * 32;
            const int *ecol = s_e + (i % 3) * kSmallN;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float part[2] = {0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int col = j * 8 + 2 * t4 + (e & 1);
                    const int erow = t.mb * 128 + r0 + 8 * (e >> 1);
                    if (col < ncol && erow < I) {
                        const float gv = acc[j][e], uv = xu[j * 4 + e], up = pow2f(ecol[col]);
                        const __half hq = __float2half_rn(__fdividef(gv * uv, 1.f + __expf(-gv * up)));
                        P.hs[(size_t)(t.pbase + col) * I + kperm_pos(erow)] = __half_as_ushort(hq);
                        part[e & 1] += __half2float(hq);
                        if (P.h_out != nullptr) {           // stage output: h of the slot
                            int f = -1;
                            if (t.shared_e) {
                                f = Tk + t.tok0 + col;
                            } else {
                                const int pos = t.pbase + col;
                                f = (pos >= 0 && pos < Tk) ? __ldg(P.perm + pos) : -1;
                                if (f >= Tk) f = -1;
                            }
                            if (f >= 0) P.h_out[(size_t)f * I + erow] = __half2float(hq) * up * up;
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) part[c] += __shfl_xor_sync(0xffffffffu, part[c], o);
                }
                if (g == 0) {
                    hp[j * 8 + 2 * t4] = part[0];
                    hp[j * 8 + 2 * t4 + 1] = part[1];
                }
            }
            __syncwarp();
            asm volatile("barrier.sync 2, %0;" ::"n"(8 * 32) : "memory");   // the eight gate warps
            const int grp = 2 * t.mb + (rw >> 2), GI = I / kGroup;
            if ((rw & 3) == 0 && lane < ncol && grp < GI) {
                const float *q4 = sH + (buf * 8 + rw) * 32 + lane;
                P.hsum[(size_t)(t.pbase + lane) * GI + grp] = ((q4[0] + q4[32]) + q4[64]) + q4[96];
            }
        }
    }
}

// ------------------------------------------------------------------ down
__global__ void __launch_bounds__(kSThreads2, 1)
    small_down_kernel(const __grid_constant__ CUtensorMap map_d, const __grid_constant__ CUtensorMap map_sd,
                      const __grid_constant__ CUtensorMap map_h, const SmallParams P)
{
    const int H = P.H, I = P.I, GI = I / kGroup, nk = GI, MB = H / 256, Tk = P.T * P.k;
    pdl_trigger();   // the tensor-memory down GEMM may take every SM this grid frees
    const int nbig = __ldg(P.nwork + 4);
    const int ntiles = (__ldg(P.nwork + 2) - nbig) * MB;
    if ((int)blockIdx.x >= ntiles) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);
    uint8_t *sC = smem;                                        // kSCodeStages x (h 4 KB | codes 2 x 4 KB)
    uint16_t *sS = reinterpret_cast<uint16_t *>(sC + kSCodeStages * 12288);  // [2][2][256][GI]
    int *s_tok = reinterpret_cast<int *>(sS + 2 * 2 * 256 * GI);             // [2][kSmallN]
    float *s_w = reinterpret_cast<float *>(s_tok + 2 * kSmallN);             // [2][kSmallN]
    const int XH = GI + 4;                 // h-sum row stride: distinct banks for the columns a warp reads
    float *s_hs = s_w + 2 * kSmallN;                                         // [2][kSmallN][XH]
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_hs + 2 * kSmallN * XH);
    uint64_t *cfull = bars, *cempty = cfull + kSCodeStages, *tfull = cempty + kSCodeStages, *tempty = tfull + 2;
    volatile int *s_abort = reinterpret_cast<volatile int *>(tempty + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kSCodeStages; ++s) {
            mbar_init(smem_u32(cfull + s), 1);
            mbar_init(smem_u32(cempty + s), kSCompute);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(tfull + b), 1 + 32);   // TMA thread (scales) + the helper warp's lanes
            mbar_init(smem_u32(tempty + b), kSCompute);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const long long limit = P.wait_limit;
    const DequantK dq = P.dq;

    if (warp == kSWarpTma) {
        // ------------------------------------------------ h boxes, code boxes, scale rows (one thread)
        if (lane != 0) return;
        prefetch_map(&map_d);
        prefetch_map(&map_sd);
        prefetch_map(&map_h);
        auto prefetch_tile = [&](int tp) {
            if (tp >= ntiles) return;
            const STile t = stile(P, nbig, tp, MB, Tk);
            const size_t wrow = (size_t)(t.shared_e ? 0 : t.expert * H) + t.mb * 256;
            prefetch_l2_bulk((t.shared_e ? P.sc0 : P.c0) + wrow * (I / 2), 256u * (I / 2));
        };
        prefetch_tile(blockIdx.x);
        int q = 0, i = 0;
        bool ok = true;
        for (int tau = blockIdx.x; tau < ntiles && ok; tau += gridDim.x, ++i) {
            const STile t = stile(P, nbig, tau, MB, Tk);
            prefetch_tile(tau + gridDim.x);
            const int buf = i & 1;
            if (i >= 2 && !mbar_wait(smem_u32(tempty + buf), ((i >> 1) - 1) & 1, limit, s_abort)) {
                set_abort(s_abort, P.status);
                break;
            }
            const size_t wrow = (size_t)(t.shared_e ? 0 : t.expert * H) + t.mb * 256;
            const uint32_t sbytes = 256u * GI * 2;
            const uint32_t tb = smem_u32(tfull + buf);
            mbar_arrive_expect_tx(tb, 2 * sbytes);
            bulk_load(smem_u32(sS + (buf * 2 + 0) * 256 * GI), (t.shared_e ? P.ss0 : P.s0) + wrow * GI, sbytes, tb);
            bulk_load(smem_u32(sS + (buf * 2 + 1) * 256 * GI), (t.shared_e ? P.sb0 : P.b0) + wrow * GI, sbytes, tb);
            const CUtensorMap *md = t.shared_e ? &map_sd : &map_d;
#pragma unroll 1
            for (int s = 0; s < nk; ++s, ++q) {
                const int cs = q % kSCodeStages;
                if (q >= kSCodeStages &&
                    !mbar_wait(smem_u32(cempty + cs), (q / kSCodeStages - 1) & 1, limit, s_abort)) {
                    set_abort(s_abort, P.status);
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(cfull + cs);
                uint8_t *stg = sC + cs * 12288;
                mbar_arrive_expect_tx(fb, 12288);
                tma_load_2d(smem_u32(stg), &map_h, s * 64, t.pbase, fb);
                tma_load_2d(smem_u32(stg + 4096), md, s * 32, (int)wrow, fb);
                tma_load_2d(smem_u32(stg + 8192), md, s * 32, (int)wrow + 128, fb);
            }
        }
        for (int d = (q > kSCodeStages ? q - kSCodeStages : 0); d < q; ++d)
            mbar_wait(smem_u32(cfull + d % kSCodeStages), (d / kSCodeStages) & 1, kSDrainLimit, nullptr);
        for (int b = 0; b < 2 && b < i; ++b) {
            const int last = i - 1 - ((i - 1 - b) & 1);
            mbar_wait(smem_u32(tfull + (last & 1)), (last >> 1) & 1, kSDrainLimit, nullptr);
        }
        return;
    }

    if (warp == kSWarpAux) {
        // ------------------------------------------------ token and weight of each column
        int i = 0;
        for (int tau = blockIdx.x; tau < ntiles; tau += gridDim.x, ++i) {
            const STile t = stile(P, nbig, tau, MB, Tk);
            const int buf = i & 1;
            // row of yslot (the column's expert-sorted position) and factor 2^2e of column `lane` (the h
            // tile holds h 2^-2e; exact)
            int tok = -1;
            float wgt = 0.f;
            if (lane < t.ntok) {
                int tt = -1;
                if (t.shared_e) {
                    tt = t.tok0 + lane;
                } else {
                    const int pos = t.pbase + lane;
                    const int f = (pos >= 0 && pos < Tk) ? __ldg(P.perm + pos) : -1;
                    if (f < 0 || f >= Tk) record_status(P.status, MOE_ERR_DEVICE);
                    else tt = f / P.k;
                }
                if (tt >= 0) {
                    const float up = pow2f(__ldg(P.xe + tt));
                    tok = t.pbase + lane;
                    wgt = up * up;
                }
            }
            bool got = i < 2 || mbar_wait(smem_u32(tempty + buf), ((i >> 1) - 1) & 1, limit, s_abort);
            got = __all_sync(0xffffffffu, got);
            if (!got) {
                set_abort(s_abort, P.status);
                break;
            }
            s_tok[buf * kSmallN + lane] = tok;
            s_w[buf * kSmallN + lane] = wgt;
            float *hsr = s_hs + (buf * kSmallN + lane) * XH;
            const float *hsg = P.hsum + (size_t)(t.pbase + lane) * GI;
#pragma unroll 1
            for (int gi = 0; gi < GI; ++gi) hsr[gi] = lane < t.ntok ? __ldg(hsg + gi) : 0.f;
            mbar_arrive(smem_u32(tfull + buf));
        }
        return;
    }

    // ---------------------------------------------------- compute warps: rows 16 w .. 16 w + 15 of 256
    const int g = lane >> 2, t4 = lane & 3;
    const int r0 = warp * 16 + g;
    int q = 0, i = 0;
    for (int tau = blockIdx.x; tau < ntiles; tau += gridDim.x, ++i) {
        const STile t = stile(P, nbig, tau, MB, Tk);
        const int buf = i & 1, ncol = t.ntok;
        bool w_ok = mbar_wait(smem_u32(tfull + buf), (i >> 1) & 1, limit, s_abort);
        const uint16_t *ssc = sS + buf * 2 * 256 * GI;
        const float *shs = s_hs + buf * kSmallN * XH;
        uint2 ws0 = make_uint2(0, 0), ws1 = ws0, wb0 = ws0, wb1 = ws0;
        float acc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
        auto step = [&](int s, int st, uint32_t par, int e) -> bool {
            if (!mbar_wait(smem_u32(cfull + st), par, limit, s_abort)) return false;
            const uint8_t *stg = sC + st * 12288;
            const uint8_t *cb = stg + 4096 + r0 * 32 + t4 * 8;
            const uint2 c0 = *reinterpret_cast<const uint2 *>(cb);
            const uint2 c1 = *reinterpret_cast<const uint2 *>(cb + 256);
            if ((e & 3) == 0) {
                ws0 = scale_window(ssc, r0, GI, s);
                ws1 = scale_window(ssc, r0 + 8, GI, s);
                wb0 = scale_window(ssc + 256 * GI, r0, GI, s);
                wb1 = scale_window(ssc + 256 * GI, r0 + 8, GI, s);
            }
            const float s0 = scale_pick(ws0, e & 3), s1 = scale_pick(ws1, e & 3);
            const float k0 = fmaf(8.f, s0, scale_pick(wb0, e & 3));
            const float k1 = fmaf(8.f, s1, scale_pick(wb1, e & 3));
            uint32_t ad[2][8];
            nib8_signed(c0.x, ad[0], dq);
            nib8_signed(c0.y, ad[0] + 4, dq);
            nib8_signed(c1.x, ad[1], dq);
            nib8_signed(c1.y, ad[1] + 4, dq);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j * 8 >= ncol) break;
                const int n = j * 8 + g;
                const uint4 lo = *reinterpret_cast<const uint4 *>(stg + swz128(n, 2 * t4));
                const uint4 hi = *reinterpret_cast<const uint4 *>(stg + swz128(n, 2 * t4 + 1));
                const uint32_t bp[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                float dd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int mm = 0; mm < 4; ++mm)
                    mma16816_f16(dd, ad[0][2 * mm], ad[1][2 * mm], ad[0][2 * mm + 1], ad[1][2 * mm + 1], bp[2 * mm],
                                 bp[2 * mm + 1]);
                const int cA = j * 8 + 2 * t4;           // h sums of the two columns over this group
                const float hA = shs[cA * XH + s], hB = shs[(cA + 1) * XH + s];
                acc[j][0] = fmaf(s0, dd[0], fmaf(k0, hA, acc[j][0]));
                acc[j][1] = fmaf(s0, dd[1], fmaf(k0, hB, acc[j][1]));
                acc[j][2] = fmaf(s1, dd[2], fmaf(k1, hA, acc[j][2]));
                acc[j][3] = fmaf(s1, dd[3], fmaf(k1, hB, acc[j][3]));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(cempty + st));
            return true;
        };
        if ((nk & 7) == 0) {
#pragma unroll 1
            for (int s8 = 0; s8 < nk && w_ok; s8 += 8) {
                const uint32_t par = ((q + s8) >> 3) & 1;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (w_ok) w_ok = step(s8 + e, e, par, e);
            }
        } else {
#pragma unroll 1
            for (int s = 0; s < nk && w_ok; ++s) w_ok = step(s, (q + s) & 7, ((q + s) >> 3) & 1, s & 7);
        }
        q += nk;
        if (!w_ok) set_abort(s_abort, P.status);
        if (compute_any(!w_ok)) {                   // all sixteen warps stop together
            set_abort(s_abort, P.status);
            break;
        }
        // y of the tile's rows and tokens into their rows of yslot (each element written once)
        const int *tok = s_tok + buf * kSmallN;
        const float *wv = s_w + buf * kSmallN;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = j * 8 + 2 * t4 + (e & 1);
                const int erow = t.mb * 256 + r0 + 8 * (e >> 1);
                if (col < ncol) {
                    const int tt = tok[col];
                    if (tt >= 0) P.yslot[(size_t)tt * H + erow] = wv[col] * acc[j][e];
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(tempty + buf));   // scales, tokens and weights no longer read
    }
}


size_t small_g1_smem(int H)
{
    const int G = H / kGroup;
    return 1024 + kG1Stages * kG1Stage + 2 * 8 * 32 * 16 * 4 + 2 * 4 * 128 * G * 2 + 2 * kSmallN * (G + 4) * 4 +
           2 * 8 * 32 * 4 + 3 * kSmallN * 4 + 8 * (2 * kG1Stages + 4) + 16;
}
size_t small_g2_smem(int I)
{
    const int GI = I / kGroup;
    return 1024 + kSCodeStages * 12288 + 2 * 2 * 256 * GI * 2 + 2 * kSmallN * 8 + 2 * kSmallN * (GI + 4) * 4 +
           8 * (2 * kSCodeStages + 4) + 16;
}

SmallParams small_params(const PrefillArgs &a, bool down)
{
    SmallParams p{};
    p.dq = kDequantK;
    p.nwork = a.nwork;
    p.work = down ? a.work_g2 : a.work_g1;
    p.offsets = a.offsets;
    p.perm = a.perm;
    p.hs = a.hs;
    p.x16 = a.x16;
    p.xsum = a.xsum;
    p.xe = a.xe;
    p.h_out = a.h_out;
    p.yslot = a.yslot;
    p.hsum = a.hsum;
    if (down) {
        p.c0 = a.down.codes;
        p.sc0 = a.has_shared ? a.s_down.codes : a.down.codes;
        p.s0 = a.down.scales;
        p.b0 = a.down.biases;
        p.ss0 = a.s_down.scales;
        p.sb0 = a.s_down.biases;
    } else {
        p.c0 = a.gate.codes;
        p.c1 = a.up.codes;
        p.sc0 = a.has_shared ? a.s_gate.codes : a.gate.codes;
        p.sc1 = a.has_shared ? a.s_up.codes : a.up.codes;
        p.s0 = a.gate.scales;
        p.b0 = a.gate.biases;
        p.s1 = a.up.scales;
        p.b1 = a.up.biases;
        p.ss0 = a.s_gate.scales;
        p.sb0 = a.s_gate.biases;
        p.ss1 = a.s_up.scales;
        p.sb1 = a.s_up.biases;
    }
    p.status = a.status;
    p.T = a.T;
    p.H = a.H;
    p.I = a.I;
    p.E = a.E;
    p.k = a.k;
    p.wait_limit = a.wait_limit;
    return p;
}

}  // namespace

// H: code rows of 128-byte... every per-tile block of scales fits the double buffer
// (H <= 2048), group-sum rows are 16-byte multiples (H % 256 == 0), whole groups in I.
bool prefill_small_fits(int H, int I, int bits)
{
    return bits == 4 && H % 256 == 0 && H <= 2048 && I % 64 == 0 && I <= 4096;
}

cudaError_t launch_small_gateup(const PrefillArgs &a, cudaStream_t st)
{
    const int H = a.H, I = a.I, E = a.E;
    CUtensorMap mg, mu, msg, msu;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapSwizzle sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
    bool ok = make_map_2d(&mg, a.gate.codes, u8, 1, H / 2, (uint64_t)E * I, 128, 128, sw128) &&
              make_map_2d(&mu, a.up.codes, u8, 1, H / 2, (uint64_t)E * I, 128, 128, sw128);
    if (a.has_shared)
        ok = ok && make_map_2d(&msg, a.s_gate.codes, u8, 1, H / 2, I, 128, 128, sw128) &&
             make_map_2d(&msu, a.s_up.codes, u8, 1, H / 2, I, 128, 128, sw128);
    else {
        msg = mg;
        msu = mu;
    }
    if (!ok) return cudaErrorInvalidValue;
    const SmallParams p = small_params(a, false);
    const size_t smem = small_g1_smem(H);
    cudaError_t e = cudaFuncSetAttribute(small_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int tiles = a.max_w1 * ((I + 127) / 128);
    small_gateup_kernel<<<std::max(1, std::min(device_sm_count(), tiles)), kSThreads1, smem, st>>>(mg, mu, msg, msu, p);
    return cudaGetLastError();
}

cudaError_t launch_small_down(const PrefillArgs &a, cudaStream_t st)
{
    const int H = a.H, I = a.I, E = a.E, T = a.T, k = a.k;
    CUtensorMap md, msd, mh;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE, sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
    bool ok = make_map_2d(&md, a.down.codes, u8, 1, I / 2, (uint64_t)E * H, 32, 128, none) &&
              make_map_2d(&mh, a.hs, f16, 2, I, (uint64_t)T * k + (uint64_t)T, 64, kSmallN, sw128);
    if (a.has_shared)
        ok = ok && make_map_2d(&msd, a.s_down.codes, u8, 1, I / 2, H, 32, 128, none);
    else
        msd = md;
    if (!ok) return cudaErrorInvalidValue;
    const SmallParams p = small_params(a, true);
    const size_t smem = small_g2_smem(I);
    cudaError_t e = cudaFuncSetAttribute(small_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int tiles = a.max_w2 * (H / 256);
    small_down_kernel<<<std::max(1, std::min(device_sm_count(), tiles)), kSThreads2, smem, st>>>(md, msd, mh, p);
    return cudaGetLastError();
}

}  // namespace qmoe
