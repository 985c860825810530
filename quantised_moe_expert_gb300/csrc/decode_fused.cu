// Fused decode layer for T <= 16: router, top-k, expert FFNs and combine in one cooperative launch.
//
// At decode sizes the layer's cost is the bytes of the selected experts (page "POC for
// qwen3.5 / qwen3.6 support optimized for AGX Orin", Phases 1-4: the batch-1 "gemv MoE
// path"; "both stacks are now weight-BW bound"): at one token ~16 MB, two or three
// microseconds of HBM time on this part.  What stands between that and the layer time is
// the chain of dependent steps (router -> top-k -> expert weights -> combine), so the
// launch is arranged to cross the grid only twice:
//
//   1. Router (every CTA, one CTA per SM).  The CTA's router rows (experts c, c + grid,
//      ...) are loaded into registers before the wait for the preceding kernel; then x is
//      staged in shared memory, the CTA's logits go to global memory tagged with the
//      launch's epoch, and x is pre-scaled per token by a power of two (x' = x 2^-e, max |x'|
//      in [1, 2), held as fp16: it keeps h inside the fp16 range, see below).  Every CTA then
//      polls the tagged logits of all tokens (all threads at once) until all carry the epoch,
//      runs the same top-k (warp max reductions, ties to the lower id), and its producer sends
//      its first unit's chunks at once, before the expert list (the same in every CTA: no
//      counter) is built.
//   2. Units.  A unit is (expert, 32-row slice s of the intermediate dimension): the
//      slice's gate and up rows (all of H) and the slice's 32 columns of the down matrix
//      (all H rows).  Because the affine rule holds for any subset of a group,
//          sum_{j in S} (s q_j + b) h_j = s sum_{j in S} q_j h_j + b sum_{j in S} h_j,
//      the CTA that computes h for its slice also applies the down projection to it at
//      once: no h crosses the grid.  A producer warp streams each unit's three chunks
//      (gate, up, down codes with the gate/up scales and biases) into a ring of shared-
//      memory slots with TMA; eight consumer warps compute them on mma.sync with the exact
//      signed codes q - 8 in fp16 (against fp16 x' for gate/up, fp16 h' for down), and write
//      per slice the raw down sums P = sum (q - 8) h' and sum h'.
//   3. One grid-wide counter; then CTA c combines rows [c RB, c RB + RB) of y: per slot,
//      y_e = 2^(2e) sum_g [ s_g (P_{2g} + P_{2g+1}) + (b_g + 8 s_g)(Hs_{2g} + Hs_{2g+1}) ],
//      then y = bf16(sum_j p_j y_ej + w_s y_shared) in slot order, one rounding.  The down
//      scales are read here, once per expert and row, in whole rows.
//
// The pick weights (fp64, one rounding to bf16) and the shared weight of token t are
// computed by CTA grid - 1 - t, off the critical path, and published before step 3.
//
// Range.  With x' = x 2^-e per token, g' = g 2^-e and u' = u 2^-e; the kernel forms
// h' = g' u' sigmoid(g' 2^e) = h 2^-2e, which is bounded by |g'||u'| whatever the size of
// x, stores it as fp16 and undoes the 2^-2e (exact) in step 3.  Rows of x far above the
// fp16 range, or entirely below its normal range, therefore lose nothing.
//
// Determinism.  Every sum has one order that depends only on the token's own data and on
// the fixed slice partition, so a token's outputs are the same bits in any batch of 1..16.
//
// Synchronisation state lives in the workspace header (two counters and an epoch); the last CTA
// to leave resets the counters and advances the epoch, so a workspace needs to be zero-filled
// only before its first use.
// Every wait is bounded (a status code is recorded instead of hanging): the waits on other CTAs by
// the caller's limit, a CTA's waits on its own copies by a fixed one (kRingLimit).
#include <mutex>
#include <type_traits>

#include "kernels.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace qmoe {
namespace {

using namespace tc;

constexpr int kCW = 8;                         // consumer warps
constexpr int kWarpProd = 8;                   // TMA producer warp
constexpr int kWarpAux = 9;                    // per-token weights and routing outputs
constexpr int kThreads = 320;
constexpr int kSlice = 32;                     // rows of the intermediate dimension per unit
constexpr int kMaxSlots = 6;
constexpr int kMaxCols = kDecodeMaxTok * (kMaxTopK + 1);
constexpr int kMaxList = kMaxExperts + 1;
// Waits on this CTA's own copies (the ring's full and empty phases, the drain) are bounded by a
// fixed number of polls, about a second: they end early only if the copy engine fails.  The
// caller's limit (moe_config.wait_polls) bounds the waits on other CTAs: the published logits and
// the unit counter.  So a small caller limit never abandons the ring with copies in flight.
constexpr long long kDrainLimit = 1ll << 22;
constexpr long long kRingLimit = 1ll << 20;
// Staged x: each group of 64 inputs padded to 72 elements and each token row by 8 more, so that
// neither lanes reading different groups (router) nor lanes reading different tokens (MMA B
// fragments) meet in one shared-memory bank.
constexpr int kXG = 72;

// Timeline stamps (trace columns), in the order a CTA reaches them.
enum {
    kStStart = 0, kStRouterPub, kStLogitsSeen, kStXStaged, kStTopk, kStListed, kStRouted, kStFirstGate,
    kStFirstDown, kStFirstDownDone, kStUnitsDone, kStUnitsCnt, kStCombineLoads, kStCombined
};

struct FusedMaps {
    CUtensorMap g, u, sg, su;   // int4 codes of gate and up (routed stacks, shared expert): 3D, 32-row boxes
};

struct FusedGeom {
    DequantK dq;        // code conversion constants (nib8_signed)
    int R;              // ring slots
    uint32_t slot;      // bytes per slot (multiple of 1024)
    uint32_t codes1;    // code bytes of a gate/up chunk: 32 rows x H / 2
    uint32_t sc1;       // bytes of its scales (and of its biases): 32 x H / 64 x 2
    uint32_t codes2;    // bytes of a down chunk: H rows x 16
    uint32_t x_off, xs_off, red_off, h_off, hs_off, dyn;
    int RB;             // rows of y combined per CTA (multiple of 4)
};

struct FSmem {
    int ids[kDecodeMaxTok][kMaxTopK];
    float lg[kDecodeMaxTok][kMaxTopK];      // fp32 logit of each pick
    float p[kDecodeMaxTok][kMaxTopK];
    float ws[kDecodeMaxTok];
    int xe[kDecodeMaxTok];                  // x' = x 2^-xe
    uint32_t pickmap[kMaxExperts / 32];     // experts picked by any token (bit e)
    uint32_t tokmask[kMaxExperts];          // tokens that picked expert e (bit t)
    int lpos[kMaxList];                     // list position of each picked expert
    int list[kMaxList];
    int ncols[kMaxList];
    int colptr[kMaxList + 1];
    int colof[kDecodeMaxTok][kMaxTopK + 1]; // column of (t, j); j == k: the shared slot
    int ctok[kMaxCols];                     // token of each column
    int colf[kMaxCols];                     // slot index f of each column (t k + j, or T k + t)
    int scanp[kThreads / 32], scanc[kThreads / 32];   // per-warp sums of the list scans
    int nlist;
    int abort;
    int cnt_state;                          // unit counter: 0 polling, 1 complete, 2 a poll ran out
    uint32_t epoch;                         // this launch's tag on the published logits
    uint64_t full[kMaxSlots], empty[kMaxSlots];
};

template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    if constexpr (F16)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// 8 consecutive 16-bit values -> the codes' k order (0,4,1,5,2,6,3,7).
__device__ __forceinline__ uint4 kperm8(uint4 v)
{
    uint4 o;
    o.x = prmt(v.x, v.z, 0x5410u);
    o.y = prmt(v.x, v.z, 0x7632u);
    o.z = prmt(v.y, v.w, 0x5410u);
    o.w = prmt(v.y, v.w, 0x7632u);
    return o;
}

// Position of element i in the k order of its chunk of 8.
__device__ __forceinline__ int kperm_pos(int i) { return (i & ~7) | ((i & 3) << 1) | ((i >> 2) & 1); }

// Byte offset, inside a row of a 128-byte code box, of the 8 code bytes lane (g, t4) reads for
// group q (0..3) of the box: 16-byte chunk 2q + t4/2 stored at chunk index (chunk ^ g).
__device__ __forceinline__ uint32_t swz_chunk(int q, int g, int t4)
{
    return (uint32_t)((((((q & 3) << 1) | (t4 >> 1)) ^ g) << 4) | ((t4 & 1) << 3));
}


__device__ __forceinline__ uint32_t logit_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) == 0) u = 0;        // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Called by whole warps; thread 0 writes the stamp and the warp is brought back together.
__device__ __forceinline__ void stamp(const FusedDecodeArgs &a, int i)
{
    if (a.trace && threadIdx.x == 0) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        a.trace[(size_t)blockIdx.x * kTraceStamps + i] = t;
    }
    __syncwarp();
}

// Named barrier 1 over the 256 consumer threads, and the same barrier ORing a predicate.  The
// non-aligned forms: a warp may reach them with its lanes apart (after a branch taken by lane 0
// only), and each warp is brought back together first as well.
__device__ __forceinline__ void consumer_bar()
{
    __syncwarp();
    asm volatile("barrier.sync 1, 256;" ::: "memory");
}
__device__ __forceinline__ bool consumer_any(bool pred)
{
    __syncwarp();
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// A warp-uniform bounded wait on an mbarrier phase (every lane polls; the warp agrees on the outcome).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, long long limit, int *abort)
{
    const bool ok = mbar_wait(smem_u32(bar), parity, limit, abort);
    return __all_sync(0xffffffffu, ok);
}

// x' for the MMAs of token t from its raw staged row, by one warp: lane l takes the row's 16-byte
// chunks l, l + 32, ..., the warp finds the row's largest |x|, scales by 2^-e (exact), rounds to fp16
// (max |x'| in [1, 2): exact for every element of at least 2^-17, and off by at most 2^-25 below),
// puts each chunk of 8 in the codes' k order and sums each group of 64 of the fp16 values (its 8
// chunks sit in 8 consecutive lanes: a fixed shuffle tree).
__device__ __forceinline__ void convert_row(FSmem &S, const FusedDecodeArgs &a, const uint16_t *s_xr, uint16_t *s_x,
                                            float *s_xs, int t)
{
    const int lane = threadIdx.x & 31, H = a.H, G = H / kGroup, XS = G * kXG + 8;
    constexpr int kMaxChunks = 2048 / 8 / 32;          // chunks per lane at the largest H
    const int cpl = H / 256;                            // chunks per lane
    uint4 v[kMaxChunks];
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < kMaxChunks; ++i)
        if (i < cpl) {
            const int c = lane + 32 * i;
            v[i] = *reinterpret_cast<const uint4 *>(s_xr + (size_t)t * XS + (c >> 3) * kXG + (c & 7) * 8);
            const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) mx = max(mx, max(w4[q] & 0x7FFFu, w4[q] >> 16 & 0x7FFFu));
        }
    mx = __reduce_max_sync(0xffffffffu, mx);
    const int xe = row_scale_exponent(mx);
    const float sc = pow2f(-xe);
#pragma unroll
    for (int i = 0; i < kMaxChunks; ++i)
        if (i < cpl) {
            const int c = lane + 32 * i;                // chunk of the row; its group is c / 8
            uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float lo = __uint_as_float(w[q] << 16) * sc, hi = __uint_as_float(w[q] & 0xFFFF0000u) * sc;
                const __half2 hv = __floats2half2_rn(lo, hi);
                w[q] = *reinterpret_cast<const uint32_t *>(&hv);
                const float2 hf = __half22float2(hv);
                sum += hf.x;
                sum += hf.y;
            }
            *reinterpret_cast<uint4 *>(s_x + (size_t)t * XS + (c >> 3) * kXG + (c & 7) * 8) =
                kperm8(make_uint4(w[0], w[1], w[2], w[3]));
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            if ((c & 7) == 0) s_xs[t * G + (c >> 3)] = sum;
        }
    if (lane == 0) S.xe[t] = xe;
}

// ------------------------------------------------------------------ routing (all threads)
//
// Top-k of every token from the fp32 logits (one warp per token: lane l holds the keys of
// experts l + 32 r, sorted once; each round takes the largest key, then the lowest id holding it),
// or the caller's ids; each pick is registered at once in a bitmap of the picked experts and, per
// expert, the set of tokens that picked it.  x' of every token is formed meanwhile by other warps
// (warp w converts tokens 9 - w, 19 - w before it polls tokens w, w + 10: the conversion fills the
// time the logits take to arrive).  Then the whole CTA: the distinct experts in increasing id (the
// shared expert last) and each expert's column count by block-wide scans, and the column of pick
// (t, j): the expert's first column plus the number of earlier tokens that picked the same expert.
// logits: the caller's fp32 logits, or null for the logits this launch publishes (tagged with its epoch).
template <class AfterTopk>
__device__ __forceinline__ void route_and_list(FSmem &S, const FusedDecodeArgs &a, const float *logits,
                                               const uint16_t *s_xr, uint16_t *s_x, float *s_xs, uint32_t *s_key,
                                               AfterTopk after_topk)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, E = a.E, k = a.k;
    constexpr int kW = kThreads / 32;
#pragma unroll 1
    for (int t = kW - 1 - warp; t < T; t += kW) convert_row(S, a, s_xr, s_x, s_xs, t);
    if (a.ids_in) {
#pragma unroll 1
        for (int i = tid; i < T * k; i += kThreads) {
            int e = a.ids_in[i];
            if (e < 0 || e >= E) {
                record_status(a.status, MOE_ERR_DEVICE);
                e = 0;
            }
            const int t = i / k;
            S.ids[t][i - t * k] = e;
            atomicOr(&S.pickmap[e >> 5], 1u << (e & 31));
            if (atomicOr(&S.tokmask[e], 1u << t) & (1u << t)) record_status(a.status, MOE_ERR_DEVICE);   // repeated id
        }
    } else {
        constexpr int RW = kMaxExperts / 32;
        if (!logits) {
            // logits published by the CTAs of this launch, each tagged with the launch's epoch: every thread
            // polls its entries of all T rows at once (entry tid + j kThreads) until every entry of every
            // row carries the epoch (bounded), leaving the order keys in shared memory
            const unsigned long long *lg = a.logits64;
            const int n = T * E;
            const uint32_t ep = S.epoch;
            // bit j: entry tid + j kThreads still stale; each pass issues all of the thread's loads before it
            // looks at any, so the round trips overlap
            constexpr int kPoll = (kDecodeMaxTok * kMaxExperts + kThreads - 1) / kThreads;
            auto poll_all = [&](auto np) {               // np: entries per thread, at most
                constexpr int NP = decltype(np)::value;
                uint32_t pend = 0;
#pragma unroll
                for (int j = 0; j < NP; ++j)
                    if (tid + j * kThreads < n) pend |= 1u << j;
                auto pass = [&]() {
                    unsigned long long v[NP];
#pragma unroll
                    for (int j = 0; j < NP; ++j) v[j] = (pend >> j) & 1u ? ld_relaxed_u64(lg + tid + j * kThreads) : 0ull;
#pragma unroll
                    for (int j = 0; j < NP; ++j)
                        if (((pend >> j) & 1u) && (uint32_t)(v[j] >> 32) == ep) {
                            s_key[tid + j * kThreads] = logit_key(__uint_as_float((uint32_t)v[j]));
                            pend &= ~(1u << j);
                        }
                };
                pass();
                long long polls = 1;
                while (__syncthreads_or(pend != 0)) {
                    if (polls++ >= a.wait_limit) {
                        if (tid == 0) {
                            S.abort = 1;
                            record_status(a.status, MOE_ERR_TIMEOUT);
                        }
                        break;
                    }
                    __nanosleep(32);
                    pass();
                }
            };
            if (n <= kThreads)
                poll_all(std::integral_constant<int, 1>{});
            else
                poll_all(std::integral_constant<int, kPoll>{});
            __syncthreads();                           // every key written (also after a timeout)
            stamp(a, kStLogitsSeen);
        }
#pragma unroll 1
        for (int t = warp; t < T; t += kW) {
            uint32_t key[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int e = lane + 32 * r;
                key[r] = e < E ? (logits ? logit_key(__ldcg(logits + (size_t)t * E + e)) : s_key[t * E + e]) : 0u;   // 0: below every logit
            }
            // the lane's RW (key, id) pairs sorted once, largest first (the key, then the lower id:
            // hi = 0xFFFF - e orders equal keys), by an 8-input sorting network; then each round takes
            // the warp's largest head (the key by one reduction, the id among equal keys by another)
            // and its lane pops it
            static_assert(RW == 8, "the sorting network below is for eight keys per lane");
            uint32_t hk[RW], hi[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                hk[r] = key[r];
                hi[r] = 0xFFFFu - (uint32_t)(lane + 32 * r);
            }
            auto cx = [&](int a0, int b0) {           // (hk, hi)[a0] >= (hk, hi)[b0] afterwards
                const bool sw = hk[b0] > hk[a0] || (hk[b0] == hk[a0] && hi[b0] > hi[a0]);
                const uint32_t ka = hk[a0], ia = hi[a0];
                hk[a0] = sw ? hk[b0] : ka;
                hi[a0] = sw ? hi[b0] : ia;
                hk[b0] = sw ? ka : hk[b0];
                hi[b0] = sw ? ia : hi[b0];
            };
            cx(0, 2); cx(1, 3); cx(4, 6); cx(5, 7);
            cx(0, 4); cx(1, 5); cx(2, 6); cx(3, 7);
            cx(0, 1); cx(2, 3); cx(4, 5); cx(6, 7);
            cx(2, 4); cx(3, 5);
            cx(1, 4); cx(3, 6);
            cx(1, 2); cx(3, 4); cx(5, 6);
            int pick = 0;
            float plg = 0.f;
#pragma unroll 1
            for (int j = 0; j < k; ++j) {
                const uint32_t mk = __reduce_max_sync(0xffffffffu, hk[0]);
                const uint32_t mi = __reduce_max_sync(0xffffffffu, hk[0] == mk ? hi[0] : 0u);
                if (hk[0] == mk && hi[0] == mi) {   // this lane's head is the pick: pop it
#pragma unroll
                    for (int r = 0; r < RW - 1; ++r) {
                        hk[r] = hk[r + 1];
                        hi[r] = hi[r + 1];
                    }
                    hk[RW - 1] = 0u;
                    hi[RW - 1] = 0u;
                }
                if (lane == j) {
                    pick = 0xFFFF - (int)mi;
                    plg = key_logit(mk);
                }
            }
            if (lane < k) {
                S.ids[t][lane] = pick;
                S.lg[t][lane] = plg;
            }
            // every pick registered at once, lane j pick j: the bitmap of picked experts and each
            // expert's set of tokens (a repeated id is reported)
            if (lane < k) {
                atomicOr(&S.pickmap[pick >> 5], 1u << (pick & 31));
                if (atomicOr(&S.tokmask[pick], 1u << t) & (1u << t)) record_status(a.status, MOE_ERR_DEVICE);
            }
        }
    }
    if (a.ids_in || logits) stamp(a, kStLogitsSeen);
    // the raw rows in the ring area are read for the last time above: ordered before the copies that
    // after_topk may issue into it
    fence_proxy_async_smem();
    __syncthreads();                 // ids, the pick bitmap and token sets, and x' of every token complete
    stamp(a, kStXStaged);
    stamp(a, kStTopk);
    after_topk();
    // the list of picked experts in increasing id (the shared expert last), each one's column count and
    // first column: thread e < E, two block-wide exclusive scans (picked flags, column counts)
    {
        const int picked = tid < E ? (int)((S.pickmap[tid >> 5] >> (tid & 31)) & 1u) : 0;
        const int c = picked ? __popc(S.tokmask[tid]) : 0;
        int sp = picked, sc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vp = __shfl_up_sync(0xffffffffu, sp, o), vc = __shfl_up_sync(0xffffffffu, sc, o);
            if (lane >= o) {
                sp += vp;
                sc += vc;
            }
        }
        if (lane == 31) {
            S.scanp[warp] = sp;
            S.scanc[warp] = sc;
        }
        __syncthreads();
        int bp = 0, bc = 0, np = 0, nc = 0;
#pragma unroll
        for (int w = 0; w < kW; ++w) {
            if (w < warp) {
                bp += S.scanp[w];
                bc += S.scanc[w];
            }
            np += S.scanp[w];
            nc += S.scanc[w];
        }
        if (picked) {
            const int pos = bp + sp - 1;
            S.list[pos] = tid;
            S.lpos[tid] = pos;
            S.ncols[pos] = c;
            S.colptr[pos] = bc + sc - c;
        }
        if (tid == 0) {
            int D = np;
            if (a.has_shared) {
                S.list[D] = E;
                S.ncols[D] = T;
                S.colptr[D] = nc;
                ++D;
            }
            S.colptr[D] = nc + (a.has_shared ? T : 0);
            S.nlist = D;
        }
    }
    __syncthreads();
    // the column of every pick (t, j): the expert's first column plus the earlier tokens that picked it
#pragma unroll 1
    for (int i = tid; i < T * k; i += kThreads) {
        const int t = i / k, j = i - t * k, e = S.ids[t][j];
        const int col = S.colptr[S.lpos[e]] + __popc(S.tokmask[e] & ((1u << t) - 1u));
        S.colof[t][j] = col;
        S.colf[col] = i;
        S.ctok[col] = t;
    }
    if (a.has_shared)
#pragma unroll 1
        for (int t = tid; t < T; t += kThreads) {
            const int col = S.colptr[S.nlist - 1] + t;
            S.colof[t][k] = col;
            S.colf[col] = T * k + t;
            S.ctok[col] = t;
        }
    __syncthreads();
    stamp(a, kStListed);
}

// ------------------------------------------------------------------ per-token weights (aux warp)
//
// Token t = grid - 1 - blockIdx: gamma = x . v in fp32 (lane l sums the groups l, l + 32, ...
// element by element in natural order, then a fixed shuffle tree: the router kernel's operations on
// the raw row, read from global memory since the staged one is gone by now), w_s =
// bf16(sigmoid(bf16(gamma))) and p_j = bf16(exp(l_j - l_0) / sum_i exp(l_i - l_0)) in fp64,
// published for the combining CTAs.
__device__ __forceinline__ void token_weights(FSmem &S, const FusedDecodeArgs &a)
{
    const int lane = threadIdx.x & 31, T = a.T, k = a.k, G = a.H / kGroup;
    const int t = (int)gridDim.x - 1 - (int)blockIdx.x;
    if (a.ids_in || t < 0 || t >= T) return;
    if (a.ids_out && lane < k) a.ids_out[t * k + lane] = S.ids[t][lane];
    double ex = 0.0;
    if (lane < k) ex = exp((double)S.lg[t][lane] - (double)S.lg[t][0]);
    double den = 0.0;
#pragma unroll 1
    for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, ex, j);   // fixed order j = 0..k-1
    if (lane < k) {
        const uint16_t pb = double_to_bf16_bits(ex / den);
        a.p_glob[t * k + lane] = pb;
        if (a.p_out) a.p_out[t * k + lane] = pb;
    }
    float part = 0.f;
    if (a.has_shared) {
#pragma unroll 1
        for (int grp = lane; grp < G; grp += 32) {
            const uint4 *xr = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + grp * kGroup);
            const uint4 *vp = reinterpret_cast<const uint4 *>(a.v + grp * kGroup);
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                const uint4 xv = xr[c], vv = __ldg(vp + c);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float xf = __uint_as_float((i & 1) ? (xw[i >> 1] & 0xFFFF0000u) : (xw[i >> 1] << 16));
                    const float vf = __uint_as_float((i & 1) ? (vw[i >> 1] & 0xFFFF0000u) : (vw[i >> 1] << 16));
                    part = fmaf(xf, vf, part);
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    }
    if (lane == 0) {
        uint16_t wsb = 0;
        if (a.has_shared) {
            const float gb = bf16_bits_to_float(float_to_bf16_bits(part));
            wsb = double_to_bf16_bits(1.0 / (1.0 + exp(-(double)gb)));
        }
        a.ws_glob[t] = wsb;
        if (a.ws_out) a.ws_out[t] = wsb;
    }
}

// ------------------------------------------------------------------ producer (one warp)
//
// Gate and up chunks: lane 0 waits for the slot, then one 3D TMA copy brings the 32 code rows (each
// 128-byte box in the 128-byte swizzle) and two bulk copies their scales and biases; the other
// lanes arrive.  Down chunk: the slice's 16-byte column of all H rows.  From the packed layout it
// is one contiguous block (one bulk copy); from the MLX layout it is 16 bytes of every 256-byte
// row, which the 32 lanes take in turn with 16-byte cp.async, each arriving (without a count
// increment) once its own copies have landed.  The first unit's chunks go out right after top-k,
// before the expert list is built (issue_first_unit); the loop issues the rest.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Chunk c (0 gate, 1 up, 2 down) of unit (expert e, slice s) into ring slot `slot`, by the producer
// warp; the slot is free.  The issuing lane (0) sets the expected bytes and issues the copies; the other
// lanes arrive (the MLX down layout: each lane's 16-byte cp.async pieces, arriving once they land).
__device__ __forceinline__ void issue_chunk(const FusedMaps &maps, const FusedDecodeArgs &a, const FusedGeom &geo,
                                            uint8_t *ring, uint64_t *full, int slot, int e, int s, int c, uint64_t pol)
{
    const int lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, E = a.E, G = H / kGroup, SL = I / kSlice;
    const bool shr = e == E;
    uint8_t *base = ring + (size_t)slot * geo.slot;
    const uint32_t fb = smem_u32(&full[slot]);
    const int row0 = (shr ? 0 : e * I) + s * kSlice;
    if (c < 2) {
        // gate or up chunk: one 3D copy of the 32 code rows (each 128-byte box in the 128-byte swizzle) and
        // two bulk copies of their scales and biases
        if (lane == 0) {
            const size_t so = (size_t)row0 * G;
            const QMatDev &m = c == 0 ? (shr ? a.s_gate : a.gate) : (shr ? a.s_up : a.up);
            mbar_arrive_expect_tx(fb, geo.codes1 + 2 * geo.sc1);
            tma_load_3d_hint(smem_u32(base), c == 0 ? (shr ? &maps.sg : &maps.g) : (shr ? &maps.su : &maps.u), 0, row0, 0,
                             fb, pol);
            bulk_load_hint(smem_u32(base + geo.codes1), m.scales + so, geo.sc1, fb, pol);
            bulk_load_hint(smem_u32(base + geo.codes1 + geo.sc1), m.biases + so, geo.sc1, fb, pol);
        } else {
            mbar_arrive(fb);
        }
    } else if (a.down_packed != nullptr && (!shr || a.s_down_packed != nullptr)) {
        // the slice's down codes are one contiguous block of the packed layout: one bulk copy
        if (lane == 0) {
            const uint8_t *src = shr ? a.s_down_packed + (size_t)s * H * 16 : a.down_packed + ((size_t)e * SL + s) * H * 16;
            mbar_arrive_expect_tx(fb, (uint32_t)H * 16);
            bulk_load_hint(smem_u32(base), src, (uint32_t)H * 16, fb, pol);
        } else {
            mbar_arrive(fb);
        }
    } else {
        const uint8_t *src = (shr ? a.s_down.codes : a.down.codes) + (size_t)(shr ? 0 : e) * H * ((size_t)I / 2) + s * 16;
        const uint32_t dst = smem_u32(base);
#pragma unroll 4
        for (int r = lane; r < H; r += 32) cp_async16(dst + r * 16, src + (size_t)r * (I / 2));
        cp_async_mbar_arrive_noinc(fb);
    }
}

// List entry d and slice s of unit u.  Units go round-robin over the CTAs (CTA b takes u = b, b + grid,
// ...), so the CTAs b < U mod grid take one unit more than the others.  The shared expert's units (a
// column per token: the heaviest) take the positions of the last full round's final CTAs, which take no
// extra unit; the routed experts' units fill the other positions in list order.
__device__ __forceinline__ void unit_at(int u, int U, int SL, int nlist, int has_shared, int &d, int &s)
{
    int v = u;
    if (has_shared) {
        const int grid = (int)gridDim.x;
        const int P = max(0, min(U - SL, (U / grid) * grid - SL));
        if (u >= P && u < P + SL) {
            d = nlist - 1;
            s = u - P;
            return;
        }
        if (u >= P + SL) v = u - SL;
    }
    d = v / SL;
    s = v - d * SL;
}

// Issued right after top-k, by the producer warp, before the expert list is built: the three chunks of this
// CTA's first unit.  The list holds the picked experts in increasing id (the shared expert last), so list
// entry d is the (d+1)-th set bit of the pick bitmap.  Returns the number of chunks issued (0 or 3).
__device__ __forceinline__ int issue_first_unit(FSmem &S, const FusedMaps &maps, const FusedDecodeArgs &a,
                                                const FusedGeom &geo, uint8_t *ring)
{
    const int lane = threadIdx.x & 31, SL = a.I / kSlice;
    constexpr int NW = kMaxExperts / 32;
    const uint32_t wbits = lane < NW ? S.pickmap[lane] : 0u;
    const int cnt = __popc(wbits);
    int pre = cnt;                                   // inclusive prefix count over the bitmap words
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, pre, o);
        if (lane >= o) pre += v;
    }
    const int npick = __shfl_sync(0xffffffffu, pre, 31);
    const int nlist = npick + (a.has_shared ? 1 : 0);
    const int u = blockIdx.x;
    if (u >= nlist * SL) return 0;
    int d, s;
    unit_at(u, nlist * SL, SL, nlist, a.has_shared, d, s);
    int e = a.E;                                     // the shared expert, last
    if (d < npick) {
        const int wl = __ffs(__ballot_sync(0xffffffffu, pre > d)) - 1;
        const uint32_t w = __shfl_sync(0xffffffffu, wbits, wl);
        const int before = __shfl_sync(0xffffffffu, pre - cnt, wl);
        e = wl * 32 + (int)__fns(w, 0, d - before + 1);
    }
    const uint64_t pol = l2_evict_first_policy();
#pragma unroll 1
    for (int c = 0; c < 3; ++c) issue_chunk(maps, a, geo, ring, S.full, c, e, s, c, pol);
    return 3;
}

// Every issued copy lands before the CTA may leave: a slot is refilled only after the warps that read it
// saw its previous copy land, so the copies still in flight are among the last R issued.
__device__ __forceinline__ void producer_drain(FSmem &S, const FusedGeom &geo, int issued)
{
    const int R = geo.R;
    if ((threadIdx.x & 31) == 0)
#pragma unroll 1
        for (int q = issued > R ? issued - R : 0; q < issued; ++q)
            mbar_wait(smem_u32(&S.full[q % R]), (q / R) & 1, kDrainLimit, nullptr);
    __syncwarp();
}

// The producer loop: units blockIdx.x, + grid, ...; the first unit's chunks may already be in flight
// (`issued` of them, from issue_first_unit).
__device__ __forceinline__ void fused_producer(FSmem &S, const FusedMaps &maps, const FusedDecodeArgs &a,
                                            const FusedGeom &geo, uint8_t *ring, int U, int issued)
{
    const int lane = threadIdx.x & 31;
    const int E = a.E, SL = a.I / kSlice, R = geo.R;
    const long long limit = kRingLimit;
    bool stop = false;
    // every weight byte is read once per launch: evict-first in L2, so the per-slice partial sums that
    // the combine reads back stay there
    const uint64_t pol = l2_evict_first_policy();
    const int i0 = issued / 3;
#pragma unroll 1
    for (int u = blockIdx.x + i0 * (int)gridDim.x, i = i0; u < U && !stop; u += gridDim.x, ++i) {
        int d, s;
        unit_at(u, U, SL, S.nlist, a.has_shared, d, s);
        const int e = S.list[d];
        if (e < 0 || e > E || d >= S.nlist) {           // a list entry out of range: report, issue nothing
            if (lane == 0) {
                S.abort = 1;
                record_status(a.status, MOE_ERR_DEVICE);
            }
            break;
        }
#pragma unroll 1
        for (int c = 0; c < 3; ++c) {
            const int q = 3 * i + c, slot = q % R;
            bool ok = true;
            if (lane == 0 && q >= R &&
                !mbar_wait(smem_u32(&S.empty[slot]), ((q / R) - 1) & 1, limit, &S.abort)) {
                S.abort = 1;
                record_status(a.status, MOE_ERR_TIMEOUT);
                ok = false;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                stop = true;
                break;
            }
            issue_chunk(maps, a, geo, ring, S.full, slot, e, s, c, pol);
            issued = q + 1;
        }
    }
    producer_drain(S, geo, issued);
}

// ------------------------------------------------------------------ consumers (warps 0-7)
//
// Gate and up chunks: warp w takes the 16-row tile mt = w % 2 and quarter kq = w / 2 of the groups of
// both matrices, with every group's product s (sum (q - 8) x') + (b + 8 s) sum x' added in
// increasing group order; the four quarters are added in order in h = silu(g) u.  Down chunk:
// warp w takes H / 128 tiles of 16 rows, K = 32 (the slice), raw sums P = sum (q - 8) h'.  The
// codes enter the MMAs signed: with 1024 + q a sum would carry ~1024 sum x' (or h') and cancel about
// eight bits against the bias term, beyond what the tensor cores' fp32 accumulation keeps.
// Element e (0..7, a compile-time index after unrolling) of eight bf16 packed in a uint4, as fp32.
__device__ __forceinline__ float bf16_of8(uint4 v, int e)
{
    const uint32_t w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

template <int NT>
__device__ __forceinline__ void fused_consumers(FSmem &S, const FusedDecodeArgs &a, const FusedGeom &geo,
                                                const uint8_t *ring, const uint16_t *s_x, const float *s_xs,
                                                float *s_red, uint16_t *s_h, float *s_hs, int U)
{
    constexpr int NC = NT * 8;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int T = a.T, H = a.H, I = a.I, G = H / kGroup, SL = I / kSlice, R = geo.R;
    const int mt = warp & 1, kq = warp >> 1, gq = G / 4, XS = G * kXG + 8;
    const long long limit = kRingLimit;
    const DequantK dq = geo.dq;
    float *const part = a.part;
    float *const hsum = a.hsum;
    bool fail_d = false;
#pragma unroll 1
    for (int u = blockIdx.x, i = 0; u < U; u += gridDim.x, ++i) {
        int d, s;
        unit_at(u, U, SL, S.nlist, a.has_shared, d, s);
        const int ncol = min(S.ncols[d], T), colbase = S.colptr[d];
        // the x' row and the group-sum rows of the lane's B column (c) and D columns (cA, cA + 1); a lane
        // whose column is past the expert's reads the first column's token instead (those MMA columns and
        // sums are never read), so every lane runs the same loads
        const int tok0 = S.ctok[colbase];
        const uint16_t *xq[NT];
        const float *xa[NT], *xb[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int c = j * 8 + g, cA = j * 8 + 2 * t4;
            xq[j] = s_x + (size_t)(c < ncol ? S.ctok[colbase + c] : tok0) * XS + 16 * t4;
            xa[j] = s_xs + (cA < ncol ? S.ctok[colbase + cA] : tok0) * G;
            xb[j] = s_xs + (cA + 1 < ncol ? S.ctok[colbase + cA + 1] : tok0) * G;
        }
        // the gate and up chunks in one pass, by all eight warps: warp w takes the 16-row tile mt = w % 2
        // and the groups of quarter kq = w / 2 of the input dimension of both matrices, so each x
        // fragment and group sum serves both and the two MMA chains interleave
        const int qg = 3 * i, qu = qg + 1, slotg = qg % R, slotu = qu % R;
        bool ok = !fail_d && warp_wait(&S.full[slotg], (qg / R) & 1, limit, &S.abort);
        if (i == 0) stamp(a, kStFirstGate);
        ok = ok && warp_wait(&S.full[slotu], (qu / R) & 1, limit, &S.abort);
        // the unit's token columns in one 8-column MMA tile (every routed expert at these sizes) or two
        // (ncol > 8): each a separate straight-line path, no per-step branch on the column count
        auto gateup = [&](auto ntu) {
            constexpr int NTU = decltype(ntu)::value;
            const uint8_t *chg = ring + (size_t)slotg * geo.slot, *chu = ring + (size_t)slotu * geo.slot;
            const uint8_t *cbg = chg + (mt * 16 + g) * 128, *cbu = chu + (mt * 16 + g) * 128;   // row mt 16 + g of every 4 KB box
            const uint16_t *scg = reinterpret_cast<const uint16_t *>(chg + geo.codes1) + (mt * 16 + g) * G;
            const uint16_t *scu = reinterpret_cast<const uint16_t *>(chu + geo.codes1) + (mt * 16 + g) * G;
            const uint16_t *big = scg + kSlice * G, *biu = scu + kSlice * G;
            float accg[NTU][4], accu[NTU][4];
#pragma unroll
            for (int j = 0; j < NTU; ++j)
#pragma unroll
                for (int v = 0; v < 4; ++v) accg[j][v] = accu[j][v] = 0.f;
            // one group: the code words of rows g, g + 8 of both matrices, the x' fragment at element xo of
            // the lane's row, the group sums at index so, the group's scales s and offsets b + 8 s
            // (sum (s q + b) x' = s sum (q - 8) x' + (b + 8 s) sum x')
            auto group_step = [&](uint2 cg0, uint2 cg1, uint2 cu0, uint2 cu1, int xo, int so, float sg0, float sg1,
                                  float kg0, float kg1, float su0, float su1, float ku0, float ku1) {
                uint32_t ag0[8], ag1[8], au0[8], au1[8];
                nib8_signed(cg0.x, ag0, dq);
                nib8_signed(cg0.y, ag0 + 4, dq);
                nib8_signed(cg1.x, ag1, dq);
                nib8_signed(cg1.y, ag1 + 4, dq);
                nib8_signed(cu0.x, au0, dq);
                nib8_signed(cu0.y, au0 + 4, dq);
                nib8_signed(cu1.x, au1, dq);
                nib8_signed(cu1.y, au1 + 4, dq);
#pragma unroll
                for (int j = 0; j < NTU; ++j) {
                    const uint4 *xr = reinterpret_cast<const uint4 *>(xq[j] + xo);
                    const uint4 lo = xr[0], hi = xr[1];
                    const uint32_t bp[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int mm = 0; mm < 4; ++mm) {
                        mma16816<true>(dg, ag0[2 * mm], ag1[2 * mm], ag0[2 * mm + 1], ag1[2 * mm + 1], bp[2 * mm],
                                       bp[2 * mm + 1]);
                        mma16816<true>(du, au0[2 * mm], au1[2 * mm], au0[2 * mm + 1], au1[2 * mm + 1], bp[2 * mm],
                                       bp[2 * mm + 1]);
                    }
                    const float xA = xa[j][so], xB = xb[j][so];
                    accg[j][0] = fmaf(sg0, dg[0], fmaf(kg0, xA, accg[j][0]));
                    accg[j][1] = fmaf(sg0, dg[1], fmaf(kg0, xB, accg[j][1]));
                    accg[j][2] = fmaf(sg1, dg[2], fmaf(kg1, xA, accg[j][2]));
                    accg[j][3] = fmaf(sg1, dg[3], fmaf(kg1, xB, accg[j][3]));
                    accu[j][0] = fmaf(su0, du[0], fmaf(ku0, xA, accu[j][0]));
                    accu[j][1] = fmaf(su0, du[1], fmaf(ku0, xB, accu[j][1]));
                    accu[j][2] = fmaf(su1, du[2], fmaf(ku1, xA, accu[j][2]));
                    accu[j][3] = fmaf(su1, du[3], fmaf(ku1, xB, accu[j][3]));
                }
            };
            // the two-tile path (the shared expert's units at T > 8, a few per launch) takes the compact
            // loop: a second fully unrolled copy would crowd the instruction cache of the hot path
            if ((gq & 7) == 0 && NTU == 1) {
                // blocks of eight groups (g0 a multiple of 8): the lane's four code offsets inside a box row
                // (group position q = 0..3) are fixed, so every load of the block is a base plus a constant.
                // Scales and biases of the eight groups per 16-byte load: rows g and g + 8 sit 64 bytes
                // apart per 32 groups, so each 2-byte load would meet three other rows in its bank.
                uint32_t swz[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) swz[q] = swz_chunk(q, g, t4);
#pragma unroll 1
                for (int gb = 0; gb < gq; gb += 8) {
                    const int g0 = kq * gq + gb;
                    const uint8_t *bg = cbg + (g0 >> 2) * (kSlice * 128), *bu = cbu + (g0 >> 2) * (kSlice * 128);
                    const uint4 vsg0 = *reinterpret_cast<const uint4 *>(scg + g0);
                    const uint4 vsg1 = *reinterpret_cast<const uint4 *>(scg + 8 * G + g0);
                    const uint4 vbg0 = *reinterpret_cast<const uint4 *>(big + g0);
                    const uint4 vbg1 = *reinterpret_cast<const uint4 *>(big + 8 * G + g0);
                    const uint4 vsu0 = *reinterpret_cast<const uint4 *>(scu + g0);
                    const uint4 vsu1 = *reinterpret_cast<const uint4 *>(scu + 8 * G + g0);
                    const uint4 vbu0 = *reinterpret_cast<const uint4 *>(biu + g0);
                    const uint4 vbu1 = *reinterpret_cast<const uint4 *>(biu + 8 * G + g0);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint32_t o = (uint32_t)(e >> 2) * (kSlice * 128) + swz[e & 3];
                        const uint2 cg0 = *reinterpret_cast<const uint2 *>(bg + o), cg1 = *reinterpret_cast<const uint2 *>(bg + o + 1024);
                        const uint2 cu0 = *reinterpret_cast<const uint2 *>(bu + o), cu1 = *reinterpret_cast<const uint2 *>(bu + o + 1024);
                        const float sg0 = bf16_of8(vsg0, e), sg1 = bf16_of8(vsg1, e);
                        const float su0 = bf16_of8(vsu0, e), su1 = bf16_of8(vsu1, e);
                        group_step(cg0, cg1, cu0, cu1, (g0 + e) * kXG, g0 + e, sg0, sg1, fmaf(8.f, sg0, bf16_of8(vbg0, e)),
                                   fmaf(8.f, sg1, bf16_of8(vbg1, e)), su0, su1, fmaf(8.f, su0, bf16_of8(vbu0, e)),
                                   fmaf(8.f, su1, bf16_of8(vbu1, e)));
                    }
                }
            } else {
#pragma unroll 2
                for (int gi = 0; gi < gq; ++gi) {
                    const int grp = kq * gq + gi;
                    const uint32_t o = (uint32_t)(grp >> 2) * (kSlice * 128) + swz_chunk(grp & 3, g, t4);
                    const uint2 cg0 = *reinterpret_cast<const uint2 *>(cbg + o), cg1 = *reinterpret_cast<const uint2 *>(cbg + o + 1024);
                    const uint2 cu0 = *reinterpret_cast<const uint2 *>(cbu + o), cu1 = *reinterpret_cast<const uint2 *>(cbu + o + 1024);
                    const float sg0 = bf16_bits_to_float(scg[grp]), sg1 = bf16_bits_to_float(scg[8 * G + grp]);
                    const float su0 = bf16_bits_to_float(scu[grp]), su1 = bf16_bits_to_float(scu[8 * G + grp]);
                    group_step(cg0, cg1, cu0, cu1, grp * kXG, grp, sg0, sg1, fmaf(8.f, sg0, bf16_bits_to_float(big[grp])),
                               fmaf(8.f, sg1, bf16_bits_to_float(big[8 * G + grp])), su0, su1,
                               fmaf(8.f, su0, bf16_bits_to_float(biu[grp])),
                               fmaf(8.f, su1, bf16_bits_to_float(biu[8 * G + grp])));
                }
            }
            // column-major [NC][32 rows]: the h step below reads one column's 32 rows, one per lane
            float *redg = s_red + (size_t)(0 * 4 + kq) * NC * kSlice + mt * 16;
            float *redu = s_red + (size_t)(1 * 4 + kq) * NC * kSlice + mt * 16;
#pragma unroll
            for (int j = 0; j < NTU; ++j) {
                const int c0 = j * 8 + 2 * t4;
                redg[c0 * kSlice + g] = accg[j][0];
                redg[(c0 + 1) * kSlice + g] = accg[j][1];
                redg[c0 * kSlice + g + 8] = accg[j][2];
                redg[(c0 + 1) * kSlice + g + 8] = accg[j][3];
                redu[c0 * kSlice + g] = accu[j][0];
                redu[(c0 + 1) * kSlice + g] = accu[j][1];
                redu[c0 * kSlice + g + 8] = accu[j][2];
                redu[(c0 + 1) * kSlice + g + 8] = accu[j][3];
            }
        };
        if (ok) {
            if (NT == 2 && ncol > 8)
                gateup(std::integral_constant<int, NT>{});
            else
                gateup(std::integral_constant<int, 1>{});
        }
        // a warp releases the chunks only once both have landed (its waits succeeded): otherwise the
        // producer could issue the next copy into a slot whose copy is still in flight
        __syncwarp();
        if (lane == 0 && ok) {
            mbar_arrive(smem_u32(&S.empty[slotg]));
            mbar_arrive(smem_u32(&S.empty[slotu]));
        }
        if (!ok && lane == 0) {
            S.abort = 1;
            record_status(a.status, MOE_ERR_TIMEOUT);
        }
        if (consumer_any(!ok)) break;

        // h' = g' u' sigmoid(g' 2^e) for the slice's 32 rows, as fp16 in the codes' k order, and its sum
#pragma unroll 1
        for (int c = warp; c < ncol; c += kCW) {
            const int row = lane;
            float gs = s_red[((0 * 4 + 0) * NC + c) * kSlice + row], us = s_red[((4 + 0) * NC + c) * kSlice + row];
#pragma unroll
            for (int v = 1; v < 4; ++v) {
                gs += s_red[((0 * 4 + v) * NC + c) * kSlice + row];
                us += s_red[((4 + v) * NC + c) * kSlice + row];
            }
            const int t = S.ctok[colbase + c];
            const float hv = gs / (1.f + __expf(-gs * pow2f(S.xe[t]))) * us;
            const __half hb = __float2half_rn(hv);
            s_h[c * kSlice + kperm_pos(row)] = __half_as_ushort(hb);
            const float hf = __half2float(hb);
            float sum = hf;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) {
                s_hs[c] = sum;
                hsum[(size_t)(colbase + c) * SL + s] = sum;
            }
            if (a.h_out) {
                const float up = pow2f(S.xe[t]);
                a.h_out[(size_t)S.colf[colbase + c] * I + s * kSlice + row] = hf * up * up;
            }
        }
        consumer_bar();

        const int q2 = 3 * i + 2, slot2 = q2 % R;
        const bool okd = warp_wait(&S.full[slot2], (q2 / R) & 1, limit, &S.abort);
        if (i == 0) stamp(a, kStFirstDown);
        auto down = [&](auto ntu) {
            constexpr int NTU = decltype(ntu)::value;
            const uint8_t *dch = ring + (size_t)slot2 * geo.slot;
            uint32_t hb[NTU][4];
#pragma unroll
            for (int j = 0; j < NTU; ++j) {
                const int c = j * 8 + g;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (c < ncol) v = *reinterpret_cast<const uint4 *>(s_h + c * kSlice + 8 * t4);
                hb[j][0] = v.x;
                hb[j][1] = v.y;
                hb[j][2] = v.z;
                hb[j][3] = v.w;
            }
            const int MT = H / (16 * kCW);
            float *pbase = part + (size_t)colbase * SL * H + (size_t)s * H;
            // one 16-row tile: independent of the others, and straight-line code (no branch: every
            // expert has a first column), so the scheduler overlaps the tiles' loads, conversions and
            // MMA chains
            auto tile = [&](int tt) {
                const int r0 = (warp * MT + tt) * 16 + g;
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(dch + r0 * 16 + 4 * t4);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(dch + (r0 + 8) * 16 + 4 * t4);
                uint32_t a0[4], a1[4];
                nib8_signed(w0, a0, dq);
                nib8_signed(w1, a1, dq);
#pragma unroll
                for (int j = 0; j < NTU; ++j) {
                    float dd[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816<true>(dd, a0[0], a1[0], a0[1], a1[1], hb[j][0], hb[j][1]);
                    mma16816<true>(dd, a0[2], a1[2], a0[3], a1[3], hb[j][2], hb[j][3]);
                    const int cA = j * 8 + 2 * t4;
                    if (cA < ncol) {
                        float *pc = pbase + (size_t)cA * SL * H;
                        pc[r0] = dd[0];
                        pc[r0 + 8] = dd[2];
                    }
                    if (cA + 1 < ncol) {
                        float *pc = pbase + (size_t)(cA + 1) * SL * H;
                        pc[r0] = dd[1];
                        pc[r0 + 8] = dd[3];
                    }
                }
            };
            if (MT == 16 && NTU == 1) {   // H = 2048: all sixteen tiles unrolled (the two-tile path stays compact)
#pragma unroll
                for (int tt = 0; tt < 16; ++tt) tile(tt);
            } else {
#pragma unroll 4
                for (int tt = 0; tt < MT; ++tt) tile(tt);
            }
        };
        if (okd) {
            if (NT == 2 && ncol > 8)
                down(std::integral_constant<int, NT>{});
            else
                down(std::integral_constant<int, 1>{});
        }
        __syncwarp();
        if (i == 0) stamp(a, kStFirstDownDone);
        if (lane == 0 && okd) mbar_arrive(smem_u32(&S.empty[slot2]));
        if (!okd && lane == 0) {
            S.abort = 1;
            record_status(a.status, MOE_ERR_TIMEOUT);
        }
        fail_d = !okd;
    }
}

// ------------------------------------------------------------------ combine (all threads)
//
// Rows [blockIdx RB, blockIdx RB + RB) of every token.  Per (token, 4 rows, slot): the slot's
// expert output y_e = 2^(2e) sum over groups, in order, of s (P_{2g} + P_{2g+1}) + (b + 8 s)
// (Hs_{2g} + Hs_{2g+1}); then per (token, 4 rows): y = sum_j p_j y_ej + w_s y_s in slot order, one
// rounding (or added to acc).  An item's loads are all issued before its first add.
__device__ __forceinline__ void fused_combine(FSmem &S, const FusedDecodeArgs &a, const FusedGeom &geo, float4 *s_t)
{
    const int tid = threadIdx.x;
    const int T = a.T, H = a.H, I = a.I, k = a.k, GI = I / kGroup, SL = I / kSlice;
    const int NS = k + (a.has_shared ? 1 : 0);
    const int r0 = (int)blockIdx.x * geo.RB;
    const int nrows = min(geo.RB, H - r0);
    if (nrows <= 0) {
        stamp(a, kStCombineLoads);
        return;
    }
    const int nq = nrows / 4;
    // the pick and shared weights (published by other CTAs): loaded now, one per thread, and stored to shared
    // memory only after the items' loads are out, so the two sets of loads share one round trip
    static_assert(kDecodeMaxTok * kMaxTopK <= kThreads, "one pick weight per thread");
    uint16_t pb = 0, wb = 0;
    if (tid < T * k) pb = a.ids_in ? a.p_in[tid] : __ldcg(a.p_glob + tid);
    if (tid < T && a.has_shared) wb = a.ids_in ? (a.ws_in ? a.ws_in[tid] : (uint16_t)0) : __ldcg(a.ws_glob + tid);
    const int nitem = T * nq * NS;
    // item it: the quad q varies fastest, so the threads of one (token, slot) read the 4 nq consecutive
    // rows of each slice's partial sums (and of the scale and bias rows) as one contiguous block
#pragma unroll 1
    for (int it = tid; it < nitem; it += kThreads) {
        const int q = it % nq, rest = it / nq, j = rest % NS, t = rest / NS;
        const int sidx = (t * nq + q) * NS + j;          // slot-order position of the item's terms
        const bool shr = j == k;
        const int e = shr ? 0 : S.ids[t][j];
        const int col = S.colof[t][j];
        const int r = r0 + 4 * q;
        if (e < 0 || e >= a.E || col < 0 || col >= S.colptr[S.nlist]) {   // out of range: report, skip
            record_status(a.status, MOE_ERR_DEVICE);
            s_t[sidx] = make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        const QMatDev &dm = shr ? a.s_down : a.down;
        const uint16_t *sp = dm.scales + ((size_t)e * H + r) * GI;
        const uint16_t *bp = dm.biases + ((size_t)e * H + r) * GI;
        const float *pp = a.part + (size_t)col * SL * H + r;
        const float *hp = a.hsum + (size_t)col * SL;
        float ye[4] = {0.f, 0.f, 0.f, 0.f};
        if (GI == 8) {
            // every load of the item first: 16 slices of 4 rows, 16 sums of h', the 4 rows' scales and biases
            float4 pv[16];
#pragma unroll
            for (int v = 0; v < 16; ++v) pv[v] = __ldcg(reinterpret_cast<const float4 *>(pp + (size_t)v * H));
            float4 hv[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) hv[v] = __ldcg(reinterpret_cast<const float4 *>(hp) + v);
            uint4 sv[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                sv[i] = __ldg(reinterpret_cast<const uint4 *>(sp) + i);
                bv[i] = __ldg(reinterpret_cast<const uint4 *>(bp) + i);
            }
            const float hsl[16] = {hv[0].x, hv[0].y, hv[0].z, hv[0].w, hv[1].x, hv[1].y, hv[1].z, hv[1].w,
                                   hv[2].x, hv[2].y, hv[2].z, hv[2].w, hv[3].x, hv[3].y, hv[3].z, hv[3].w};
#pragma unroll
            for (int gg = 0; gg < 8; ++gg) {
                const float hs = hsl[2 * gg] + hsl[2 * gg + 1];
                const float4 p0 = pv[2 * gg], p1 = pv[2 * gg + 1];
                const float ps[4] = {p0.x + p1.x, p0.y + p1.y, p0.z + p1.z, p0.w + p1.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t sw = gg < 2 ? sv[i].x : gg < 4 ? sv[i].y : gg < 6 ? sv[i].z : sv[i].w;
                    const uint32_t bw = gg < 2 ? bv[i].x : gg < 4 ? bv[i].y : gg < 6 ? bv[i].z : bv[i].w;
                    const float sc = __uint_as_float((gg & 1) ? (sw & 0xFFFF0000u) : (sw << 16));
                    const float bi = __uint_as_float((gg & 1) ? (bw & 0xFFFF0000u) : (bw << 16));
                    ye[i] += fmaf(sc, ps[i], fmaf(8.f, sc, bi) * hs);
                }
            }
        } else {
#pragma unroll 4
            for (int gg = 0; gg < GI; ++gg) {
                const float4 p0 = __ldcg(reinterpret_cast<const float4 *>(pp + (size_t)(2 * gg) * H));
                const float4 p1 = __ldcg(reinterpret_cast<const float4 *>(pp + (size_t)(2 * gg + 1) * H));
                const float hs = __ldcg(hp + 2 * gg) + __ldcg(hp + 2 * gg + 1);
                const float ps[4] = {p0.x + p1.x, p0.y + p1.y, p0.z + p1.z, p0.w + p1.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float sc = bf16_bits_to_float(__ldg(sp + (size_t)i * GI + gg));
                    const float bi = bf16_bits_to_float(__ldg(bp + (size_t)i * GI + gg));
                    ye[i] += fmaf(sc, ps[i], fmaf(8.f, sc, bi) * hs);
                }
            }
        }
        const float up = pow2f(S.xe[t]);
        const float4 v = make_float4(ye[0] * up * up, ye[1] * up * up, ye[2] * up * up, ye[3] * up * up);
        s_t[sidx] = v;
        if (a.yslot_out) {
            const int f = shr ? T * k + t : t * k + j;
            *reinterpret_cast<float4 *>(a.yslot_out + (size_t)f * H + r) = v;
        }
    }
    if (tid < T * k) S.p[tid / k][tid % k] = bf16_bits_to_float(pb);
    if (tid < T) S.ws[tid] = bf16_bits_to_float(wb);
    __syncthreads();
    stamp(a, kStCombineLoads);
    if (a.stages_only) return;
#pragma unroll 1
    for (int it = tid; it < T * nq; it += kThreads) {
        const int q = it % nq, t = it / nq, r = r0 + 4 * q;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int j = 0; j < NS; ++j) {
            const float4 ye = s_t[(size_t)it * NS + j];
            const float w = j == k ? S.ws[t] : S.p[t][j];
            sum.x = fmaf(w, ye.x, sum.x);
            sum.y = fmaf(w, ye.y, sum.y);
            sum.z = fmaf(w, ye.z, sum.z);
            sum.w = fmaf(w, ye.w, sum.w);
        }
        if (a.y) {
            const uint32_t lo = (uint32_t)float_to_bf16_bits(sum.x) | ((uint32_t)float_to_bf16_bits(sum.y) << 16);
            const uint32_t hi = (uint32_t)float_to_bf16_bits(sum.z) | ((uint32_t)float_to_bf16_bits(sum.w) << 16);
            *reinterpret_cast<uint2 *>(a.y + (size_t)t * H + r) = make_uint2(lo, hi);
        } else {
            float4 *ap = reinterpret_cast<float4 *>(a.acc + (size_t)t * H + r);
            float4 av = *ap;
            av.x += sum.x;
            av.y += sum.y;
            av.z += sum.z;
            av.w += sum.w;
            *ap = av;
        }
    }
}

// Asks L2 for the down scale and bias rows this CTA combines, for every listed expert (they are
// read after the unit counter, on the critical path).  Per-thread line prefetches, not bulk ones:
// a CTA that stops early (a wait ran out) leaves soon after this, and a bulk prefetch has no
// completion the CTA could wait for, so none may still sit in the copy engine when it exits.
__device__ __forceinline__ void prefetch_combine_scales(const FSmem &S, const FusedDecodeArgs &a, const FusedGeom &geo)
{
    const int lane = threadIdx.x & 31, H = a.H, E = a.E, GI = a.I / kGroup;
    const int r0 = (int)blockIdx.x * geo.RB, nrows = min(geo.RB, H - r0);
    if (nrows <= 0) return;
    const int bytes = nrows * GI * 2, nlines = (bytes + 127) / 128;
#pragma unroll 1
    for (int d = lane; d < S.nlist; d += 32) {
        const int e = S.list[d];
        const bool shr = e == E;
        const QMatDev &dm = shr ? a.s_down : a.down;
        const size_t o = ((size_t)(shr ? 0 : e) * H + r0) * GI;
        const uint8_t *sp = reinterpret_cast<const uint8_t *>(dm.scales + o);
        const uint8_t *bp = reinterpret_cast<const uint8_t *>(dm.biases + o);
#pragma unroll 1
        for (int l = 0; l < nlines; ++l) {
            const int off = min(l * 128, bytes - 1);
            prefetch_l2_line(sp + off);
            prefetch_l2_line(bp + off);
        }
    }
}

// ------------------------------------------------------------------ kernel
template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fused_kernel(const __grid_constant__ FusedMaps maps, const __grid_constant__ FusedDecodeArgs a,
                        const __grid_constant__ FusedGeom geo)
{
    __shared__ FSmem S;
    extern __shared__ uint8_t dyn_raw[];
    uint8_t *dyn = align_smem_1024(dyn_raw);
    uint8_t *ring = dyn;
    uint16_t *s_x = reinterpret_cast<uint16_t *>(dyn + geo.x_off);    // [T][G * 72 + 8] fp16 x', k order
    float *s_xs = reinterpret_cast<float *>(dyn + geo.xs_off);         // [T][G] group sums of x'
    float *s_red = reinterpret_cast<float *>(dyn + geo.red_off);       // [2][4][NC][32]
    uint16_t *s_h = reinterpret_cast<uint16_t *>(dyn + geo.h_off);     // [NC][32] fp16 h', k order
    float *s_hs = reinterpret_cast<float *>(dyn + geo.hs_off);         // [NC]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, H = a.H, E = a.E, G = H / kGroup, SL = a.I / kSlice;
    const int grid = gridDim.x, cta = blockIdx.x;
    const long long limit = a.wait_limit;
    int *const cnt_units = a.sync + kSyncUnits, *const cnt_exit = a.sync + kSyncExit;
    stamp(a, kStStart);

    if (tid == 0) {
        for (int s = 0; s < geo.R; ++s) {
            mbar_init(smem_u32(&S.full[s]), 32);   // every producer lane arrives once per chunk
            mbar_init(smem_u32(&S.empty[s]), kCW);
        }
        S.abort = 0;
        fence_mbar_init();
    }
#pragma unroll 1
    for (int e = tid; e < kMaxExperts; e += kThreads) S.tokmask[e] = 0u;
    if (tid < kMaxExperts / 32) S.pickmap[tid] = 0u;

    // this CTA's router rows (weights only: read before the wait for the preceding kernel)
    const bool router = a.ids_in == nullptr && a.logits_in == nullptr;
    const int nre = router && cta < E ? (E - 1 - cta) / grid + 1 : 0;
    int er = -1, rt0 = 0, rstep = 1;
    uint4 rc[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                   make_uint4(0u, 0u, 0u, 0u)};
    float rs = 0.f, rbias = 0.f;
    if (nre > 0 && warp < kCW) {
        const int stride = kCW / nre;
        if (warp / nre < stride) {
            er = cta + grid * (warp % nre);
            rt0 = warp / nre;
            rstep = stride;
        }
        if (er >= 0 && lane < G) {
            const uint4 *cp = reinterpret_cast<const uint4 *>(a.r_codes + (size_t)er * H + lane * kGroup);
#pragma unroll
            for (int c = 0; c < 4; ++c) rc[c] = __ldg(cp + c);
            rs = bf16_bits_to_float(__ldg(a.r_scales + (size_t)er * G + lane));
            rbias = bf16_bits_to_float(__ldg(a.r_biases + (size_t)er * G + lane));
        }
    }
    if (warp == kWarpProd && lane == 0) {
        prefetch_map(&maps.g);
        prefetch_map(&maps.u);
        if (a.has_shared) {
            prefetch_map(&maps.sg);
            prefetch_map(&maps.su);
        }
    }

    // ---- everything below reads what the preceding kernel wrote (x, the workspace header).  Raw x
    // goes into the ring area (idle until the units start) with its groups of 64 padded to 72
    // elements, so that lanes reading different groups meet in no shared-memory bank.
    pdl_wait();
    const int XS = G * kXG + 8;
    uint16_t *s_xr = reinterpret_cast<uint16_t *>(ring);        // [T][XS] bf16 x, natural order
    {
        const int cpr = H / 8;
#pragma unroll 1
        for (int i = tid; i < T * cpr; i += kThreads) {
            const int t = i / cpr, c = i - t * cpr;
            cp_async16(smem_u32(s_xr + (size_t)t * XS + (c >> 3) * kXG + (c & 7) * 8),
                       reinterpret_cast<const uint4 *>(a.x) + i);
        }
        cp_async_commit();
    }
    uint32_t epoch = 0;
    if (lane == 0) epoch = (uint32_t)ld_acquire_gpu(a.sync + kSyncEpoch) + 1u;   // in flight with x
    if (tid == 0) S.epoch = epoch;
    cp_async_wait_all();
    __syncthreads();

    // ---- router logits of this CTA's experts: per group s sum q x + b sum x in fp32, elements in
    // order, then a fixed shuffle tree (the operations of the router kernel, on the same unscaled x),
    // published as (logit, epoch) pairs that the other CTAs poll
    if (er >= 0) {
#pragma unroll 1
        for (int t = rt0; t < T; t += rstep) {
            float prt = 0.f;
            if (lane < G) {
                const uint4 *xr = reinterpret_cast<const uint4 *>(s_xr + (size_t)t * XS + lane * kXG);
                float dq = 0.f, sx = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 xv = xr[c];
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                    const uint32_t clo = (c & 1) ? rc[c >> 1].z : rc[c >> 1].x;
                    const uint32_t chi = (c & 1) ? rc[c >> 1].w : rc[c >> 1].y;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t cw = q < 2 ? clo : chi;
                        const float q0 = (float)((cw >> ((2 * q & 3) * 8)) & 0xFFu);
                        const float q1 = (float)((cw >> (((2 * q & 3) + 1) * 8)) & 0xFFu);
                        const float x0 = __uint_as_float(xw[q] << 16), x1 = __uint_as_float(xw[q] & 0xFFFF0000u);
                        dq = fmaf(q0, x0, dq);
                        dq = fmaf(q1, x1, dq);
                        sx += x0;
                        sx += x1;
                    }
                }
                prt = fmaf(rs, dq, fmaf(rbias, sx, 0.f));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) prt += __shfl_xor_sync(0xffffffffu, prt, o);
            if (lane == 0) {
                float l = prt;
                if (a.router_bias) l = l + __ldg(a.router_bias + er);   // one fp32 rounding
                st_relaxed_u64(a.logits64 + (size_t)t * E + er, ((unsigned long long)epoch << 32) | __float_as_uint(l));
            }
        }
    }
    stamp(a, kStRouterPub);

    // ---- routing, and x' for the expert units from the raw rows in the ring area (route_and_list)
    int U = 0, early = 0;
    if (!S.abort) {
        // the producer sends the first unit's chunks as soon as the picks are known
        uint32_t *s_key = reinterpret_cast<uint32_t *>(ring + ((size_t)T * XS * 2 + 15) / 16 * 16);   // after raw x
        route_and_list(S, a, a.logits_in, s_xr, s_x, s_xs, s_key, [&]() {
            if (warp == kWarpProd && !S.abort) early = issue_first_unit(S, maps, a, geo, ring);
        });
        U = S.nlist * SL;
    }
    stamp(a, kStRouted);
    // every warp takes its role or none: the flag is read before any role may set it; the ring area is
    // handed to the copy engine after this barrier (its generic-proxy reads are ordered before it)
    const bool go = !S.abort;
    fence_proxy_async_smem();
    __syncthreads();

    if (!go && warp == kWarpProd) producer_drain(S, geo, early);   // copies already in flight land first
    if (go) {
        if (warp == kWarpProd) {
            fused_producer(S, maps, a, geo, ring, U, early);
        } else if (warp == kWarpAux) {
            prefetch_combine_scales(S, a, geo);
            token_weights(S, a);
        } else {
            fused_consumers<NT>(S, a, geo, ring, s_x, s_xs, s_red, s_h, s_hs, U);
        }
    }
    if ((int)blockIdx.x >= U) {          // no units: the first-unit stamps take this time
        stamp(a, kStFirstGate);
        stamp(a, kStFirstDown);
        stamp(a, kStFirstDownDone);
    }
    __syncthreads();
    stamp(a, kStUnitsDone);
    // the unit counter: thread 0 adds this CTA; then lane 0 of every warp polls it, their first polls spread
    // over about one L2 round trip, so the count is seen soon after it reaches L2; the first poller to see it
    // (with an acquire load) tells the others through shared memory, and the barrier orders every thread's
    // reads of the other CTAs' partial sums after that acquire
    if (tid == 0) {
        S.cnt_state = 0;
        if (!S.abort) {
            __threadfence();        // this CTA's partial sums and published weights, before the count
            const int old = atomicAdd(cnt_units, 1);
            if (old < 0 || old >= grid) {
                record_status(a.status, MOE_ERR_WORKSPACE);
                S.abort = 1;
            }
        }
    }
    __syncthreads();
    if (!S.abort && lane == 0) {
        volatile int *st = &S.cnt_state;
        __nanosleep(96 * warp);
        for (long long n = 1; *st == 0; ++n) {
            if (ld_acquire_gpu(cnt_units) >= grid) {
                *st = 1;
                break;
            }
            if (n >= limit) {
                if (atomicCAS(&S.cnt_state, 0, 2) == 0) {
                    record_status(a.status, MOE_ERR_TIMEOUT);
                    S.abort = 1;
                }
                break;
            }
            __nanosleep(32);
        }
    }
    __syncthreads();
    stamp(a, kStUnitsCnt);
    pdl_trigger();
    if (!S.abort) fused_combine(S, a, geo, reinterpret_cast<float4 *>(ring));
    __syncthreads();
    stamp(a, kStCombined);
    // the last CTA out resets the counters for the next call on this workspace
    if (tid == 0) {
        const int old = atomicAdd(cnt_exit, 1);
        if (old == grid - 1) {
            *cnt_units = 0;
            *cnt_exit = 0;
            a.sync[kSyncEpoch] = (int)S.epoch;   // the next launch tags its logits with epoch + 1
        } else if (old < 0 || old >= grid) {
            record_status(a.status, MOE_ERR_WORKSPACE);
        }
    }
}

// ------------------------------------------------------------------ host side

std::mutex g_attr_mutex;

// Cached per-device attributes (device ids 0..kMaxDev-1).
constexpr int kMaxDev = 64;
struct DevInfo {
    int sms = 0, optin = 0;
};
DevInfo g_dev[kMaxDev];
uint32_t g_smem_set[kMaxDev][2];     // largest dynamic shared-memory size set so far per kernel

bool dev_info(int dev, DevInfo *out)
{
    if (dev < 0 || dev >= kMaxDev) return false;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    DevInfo &d = g_dev[dev];
    if (d.sms == 0) {
        int sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return false;
        d.sms = sms;
        d.optin = optin;
    }
    *out = d;
    return true;
}

bool fused_geometry(int T, int H, int I, int E, int k, int has_shared, int grid, int optin, FusedGeom *out)
{
    if (T < 1 || T > kDecodeMaxTok || H % 256 || H > 2048 || I % 64 || I > 4096 || grid < 1) return false;
    FusedGeom g{};
    g.dq = kDequantK;
    const int G = H / kGroup, NT = T > 8 ? 2 : 1, NC = 8 * NT;
    g.codes1 = (uint32_t)kSlice * H / 2;
    g.sc1 = (uint32_t)kSlice * G * 2;
    g.codes2 = (uint32_t)H * 16;
    g.slot = (uint32_t)align_up(std::max(g.codes1 + 2 * g.sc1, g.codes2), 1024);
    const size_t xb = align_up((size_t)T * (G * kXG + 8) * 2, 16), xsb = align_up((size_t)T * G * 4, 16);
    const size_t redb = (size_t)2 * 4 * kSlice * NC * 4, hb = (size_t)NC * kSlice * 2, hsb = align_up((size_t)NC * 4, 16);
    const size_t fixed = xb + xsb + redb + hb + hsb;
    const long long budget = (long long)optin - (long long)sizeof(FSmem) - 1024 - 64;
    if (budget <= (long long)fixed) return false;
    long long R = (budget - (long long)fixed) / g.slot;
    if (R > kMaxSlots) R = kMaxSlots;
    if (R < 3) return false;
    g.R = (int)R;
    g.RB = 4 * ((H + 4 * grid - 1) / (4 * grid));
    const int NS = k + (has_shared ? 1 : 0);
    if ((size_t)T * (g.RB / 4) * NS * 16 > (size_t)g.R * g.slot) return false;   // combine terms in the ring
    // raw x, then the order keys of the polled logits, in the ring area
    if (((size_t)T * (G * kXG + 8) * 2 + 15) / 16 * 16 + (size_t)T * E * 4 > (size_t)g.R * g.slot) return false;
    size_t o = (size_t)g.R * g.slot;
    g.x_off = (uint32_t)o;
    o += xb;
    g.xs_off = (uint32_t)o;
    o += xsb;
    g.red_off = (uint32_t)o;
    o += redb;
    g.h_off = (uint32_t)o;
    o += hb;
    g.hs_off = (uint32_t)o;
    o += hsb;
    g.dyn = (uint32_t)(o + 1024);    // slack for aligning the base to 1024 bytes
    *out = g;
    return true;
}

bool code_map_rows(CUtensorMap *m, const uint8_t *codes, int row_bytes, uint64_t rows, int box_rows)
{
    // (128-byte chunk, row, chunk index), chunk index outermost: one copy brings every 128-byte box
    // of a unit's rows, each box landing as [box_rows][128] with the 128-byte swizzle
    const uint64_t dims[3] = {128u, rows, (uint64_t)row_bytes / 128u};
    const uint64_t strides[2] = {(uint64_t)row_bytes, 128u};
    const uint32_t box[3] = {128u, (uint32_t)box_rows, (uint32_t)row_bytes / 128u};
    return make_map_3d(m, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool decode_fused_fits(int T, int H, int I, int E, int k, int has_shared)
{
    int dev = 0;
    DevInfo di;
    if (cudaGetDevice(&dev) != cudaSuccess || !dev_info(dev, &di)) return false;
    if (E > kCW * di.sms || di.sms > kTraceMaxCtas) return false;   // at most eight router experts per CTA
    FusedGeom g;
    return fused_geometry(T, H, I, E, k, has_shared, di.sms, di.optin, &g);
}

size_t decode_fused_trace_ctas()
{
    int dev = 0;
    DevInfo di;
    if (cudaGetDevice(&dev) != cudaSuccess || !dev_info(dev, &di)) return 0;
    return (size_t)di.sms;
}

cudaError_t launch_decode_fused(const FusedDecodeArgs &a, cudaStream_t st)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    DevInfo di;
    if (!dev_info(dev, &di)) return cudaErrorInvalidDevice;
    FusedGeom geo;
    if (!fused_geometry(a.T, a.H, a.I, a.E, a.k, a.has_shared, di.sms, di.optin, &geo)) return cudaErrorInvalidValue;
    FusedMaps maps;
    const uint64_t E = (uint64_t)a.E;
    bool ok = code_map_rows(&maps.g, a.gate.codes, a.H / 2, E * a.I, kSlice) &&
              code_map_rows(&maps.u, a.up.codes, a.H / 2, E * a.I, kSlice);
    if (ok && a.has_shared)
        ok = code_map_rows(&maps.sg, a.s_gate.codes, a.H / 2, a.I, kSlice) &&
             code_map_rows(&maps.su, a.s_up.codes, a.H / 2, a.I, kSlice);
    else if (ok) {
        maps.sg = maps.g;
        maps.su = maps.u;
    }
    if (!ok) return cudaErrorInvalidValue;
    const int which = a.T > 8 ? 1 : 0;
    auto kern = which ? decode_fused_kernel<2> : decode_fused_kernel<1>;
    {
        // raised (never lowered) to the largest size a launch of this kernel on the device asks for
        std::lock_guard<std::mutex> lock(g_attr_mutex);
        if (g_smem_set[dev][which] < geo.dyn) {
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.dyn)) !=
                cudaSuccess)
                return e;
            g_smem_set[dev][which] = geo.dyn;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(di.sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = geo.dyn;
    cfg.stream = st;
    // cooperative (the CTAs wait on one another), and allowed to start while the kernel
    // before it still runs: only weights are read before the wait for it
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, maps, a, geo);
}

__global__ void __launch_bounds__(256) pack_down_kernel(const uint8_t *src, uint8_t *dst, int n, int H, int I)
{
    // one 16-byte piece per thread: (matrix m, row r, slice c) -> dst[((m * SL + c) * H + r) * 16]
    const int SL = I / kSlice;
    const size_t total = (size_t)n * H * SL;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % SL);
        const size_t mr = i / SL;
        const int r = (int)(mr % H);
        const size_t m = mr / H;
        const uint4 v = *reinterpret_cast<const uint4 *>(src + mr * (size_t)(I / 2) + (size_t)c * 16);
        *reinterpret_cast<uint4 *>(dst + ((m * SL + c) * H + r) * 16) = v;
    }
}

cudaError_t launch_pack_down(const uint8_t *src, uint8_t *dst, int n, int H, int I, cudaStream_t st)
{
    const size_t total = (size_t)n * H * (I / kSlice);
    const int blocks = (int)std::min<size_t>((total + 255) / 256, 4096);
    if (blocks == 0) return cudaSuccess;
    pack_down_kernel<<<blocks, 256, 0, st>>>(src, dst, n, H, I);
    return cudaGetLastError();
}

}  // namespace qmoe
