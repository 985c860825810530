// Router GEMV, top-k / pick weights / shared weight, and the stable permutation.
//
// Follows the routing contract of the page "Qwen3.6-35B-A3B (qwen3_5_moe) on the
// native Metal engine: proposal and gate", slice "The family, plain decode":
// fp32 logits, top-k by logit with ties to the lower id, weights exp(l - l_top)
// normalised over the picks and rounded to bf16, shared slot weight
// bf16(sigmoid(bf16(gate))).  The router is MLX affine 8-bit in groups of 64.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace qmoe {

// ---------------------------------------------------------------- router GEMV
//
// grid.x: ceil(E / 8) expert tiles plus one extra column that computes the
// shared gate logit gamma; grid.y: ceil(T / 8) token tiles.  256 threads: warp
// w owns expert (tile*8 + w) for the tile's 8 tokens.  Lane l owns the groups
// g = l, l + 32, ... of the hidden dimension; per group
//     partial += s_g * sum_j(q_j * x_j) + b_g * sum_j(x_j)
// in fp32, then a fixed shuffle tree adds the 32 lane partials.  The
// arithmetic of one token never depends on the other tokens of the tile, so a
// token's logits are the same bits at every batch size.
__global__ void __launch_bounds__(256) route_gemv_kernel(RouteArgs a)
{
    tc::pdl_trigger();   // the fused decode kernel may start its prologue (it waits before reading our outputs)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.y * 8;
    const int H = a.H, E = a.E, G = a.H / kGroup;
    const int ntok = min(8, a.T - t0);
    const bool gamma_col = (int)blockIdx.x == a.n_expert_tiles;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        if (a.status_reset && threadIdx.x == 0) *a.status_reset = 0;
        for (int i = threadIdx.x; i < a.nzero; i += blockDim.x) a.zero[i] = 0;
    }

    if (gamma_col) {
        // gamma[t] = sum_h x[t,h] * v[h] in fp32, warp w -> token t0 + w.
        if (warp >= ntok || a.v == nullptr) return;
        const int t = t0 + warp;
        float part = 0.f;
        for (int g = lane; g < G; g += 32) {
            const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + (size_t)t * H + g * kGroup);
            const uint4 *vp = reinterpret_cast<const uint4 *>(a.v + g * kGroup);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 xv = __ldg(xp + c), vv = __ldg(vp + c);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    part = fmaf(__uint_as_float(xw[q] << 16), __uint_as_float(vw[q] << 16), part);
                    part = fmaf(__uint_as_float(xw[q] & 0xFFFF0000u), __uint_as_float(vw[q] & 0xFFFF0000u), part);
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) a.gamma[t] = part;
        return;
    }

    const int e = blockIdx.x * 8 + warp;
    if (e >= E) return;
    float part[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) part[i] = 0.f;

    const uint8_t *crow = a.r_codes + (size_t)e * H;
    for (int g = lane; g < G; g += 32) {
        uint4 cq[4];
        const uint4 *cp = reinterpret_cast<const uint4 *>(crow + g * kGroup);
#pragma unroll
        for (int c = 0; c < 4; ++c) cq[c] = __ldg(cp + c);
        const float s = bf16_bits_to_float(__ldg(a.r_scales + (size_t)e * G + g));
        const float b = bf16_bits_to_float(__ldg(a.r_biases + (size_t)e * G + g));
        const uint32_t cw[16] = {cq[0].x, cq[0].y, cq[0].z, cq[0].w, cq[1].x, cq[1].y, cq[1].z, cq[1].w,
                                 cq[2].x, cq[2].y, cq[2].z, cq[2].w, cq[3].x, cq[3].y, cq[3].z, cq[3].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < ntok) {
                const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + (size_t)(t0 + i) * H + g * kGroup);
                float dq = 0.f, sx = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 xv = __ldg(xp + c);
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = c * 8 + q * 2;                  // element index within the group
                        const uint32_t codes4 = cw[j >> 2];
                        const float q0 = (float)((codes4 >> ((j & 3) * 8)) & 0xFFu);
                        const float q1 = (float)((codes4 >> (((j & 3) + 1) * 8)) & 0xFFu);
                        const float x0 = __uint_as_float(xw[q] << 16);
                        const float x1 = __uint_as_float(xw[q] & 0xFFFF0000u);
                        dq = fmaf(q0, x0, dq);
                        dq = fmaf(q1, x1, dq);
                        sx += x0;
                        sx += x1;
                    }
                }
                part[i] = fmaf(s, dq, fmaf(b, sx, part[i]));
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part[i] += __shfl_xor_sync(0xffffffffu, part[i], o);
    }
    if (lane < ntok) {
        float l = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i == lane) l = part[i];
        if (a.router_bias) l = l + __ldg(a.router_bias + e);   // one fp32 rounding
        a.logits[(size_t)(t0 + lane) * E + e] = l;
    }
}

// ---------------------------------------------------------------- top-k
//
// One warp per token, 8 tokens per block.  Lane l holds logits e = l + 32 r.
// A logit maps to an order-preserving unsigned key (+0 and -0 map to the same
// key); the pair (key, 0xFFFF - id) is maximised, so equal logits resolve to
// the lower id: each lane sorts its pairs once, then k rounds of two warp
// reductions give the ids in rank order.  Weights
// are computed in fp64 and rounded once to bf16 (fp64 is scarce on this GPU,
// hence few tokens per block so the work spreads over every SM).  Each pick
// is counted into the histogram row of its 128-token block (global atomics).
__device__ __forceinline__ uint32_t logit_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) == 0) u = 0;                  // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// bf16 rounding of a positive fp32 value v known to a few fp32 ulps: the rounded bits when v lies more
// than kBf16Margin fp32 ulps from a bf16 rounding midpoint (so the exact value rounds the same way),
// else kBf16Unclear (not a bf16 of a finite positive value below 2).  Values below 2^-100 (where an
// underflowing exp loses its relative accuracy) are always unclear.
constexpr int kBf16Margin = 64;
constexpr uint16_t kBf16Unclear = 0xFFFFu;
__device__ __forceinline__ uint16_t bf16_if_clear(float v)
{
    if (!(v >= 0x1p-100f)) return kBf16Unclear;
    const uint32_t u = __float_as_uint(v);
    const int low = (int)(u & 0xFFFFu) - 0x8000;       // distance from the midpoint in fp32 ulps
    if (low > -kBf16Margin && low < kBf16Margin) return kBf16Unclear;
    return float_to_bf16_bits(v);
}

__global__ void __launch_bounds__(256) topk_kernel(TopkArgs a)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E, k = a.k;
    const int R = (E + 31) / 32;
    {
        const int t = blockIdx.x * 8 + warp;
        if (t >= a.T) return;
        const float *lrow = a.logits + (size_t)t * E;
        uint32_t key[kMaxExperts / 32];
#pragma unroll
        for (int r = 0; r < kMaxExperts / 32; ++r) {
            const int e = lane + 32 * r;
            key[r] = r < R && e < E ? logit_key(lrow[e]) : 0u;   // 0: below every real key
        }
        // the lane's eight (key, id) pairs sorted once, largest first (the key, then the lower id: hi =
        // 0xFFFF - e orders equal keys), by an 8-input sorting network; then each round takes the warp's
        // largest head (the key by one reduction, the id among equal keys by another) and its lane pops it
        static_assert(kMaxExperts / 32 == 8, "the sorting network below is for eight keys per lane");
        uint32_t hk[8], hi[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
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
        int my_id = -1;         // lane j < k ends with the id of rank j
        float my_l = 0.f;
        float top_l = 0.f;
#pragma unroll 1
        for (int j = 0; j < k; ++j) {
            const uint32_t mk = __reduce_max_sync(0xffffffffu, hk[0]);
            const uint32_t mi = __reduce_max_sync(0xffffffffu, hk[0] == mk ? hi[0] : 0u);
            if (hk[0] == mk && hi[0] == mi) {   // this lane's head is the pick: pop it
#pragma unroll
                for (int r = 0; r < 7; ++r) {
                    hk[r] = hk[r + 1];
                    hi[r] = hi[r + 1];
                }
                hk[7] = 0u;
                hi[7] = 0u;
            }
            // the winner's logit from its key (the key map is one to one but for -0, which reads as +0)
            const float v = __uint_as_float((mk & 0x80000000u) ? (mk & 0x7FFFFFFFu) : ~mk);
            if (j == 0) top_l = v;
            if (lane == j) {
                my_id = 0xFFFF - (int)mi;
                my_l = v;
            }
        }
        // pick weights p_j = exp(l_j - l_top) / sum_i exp(l_i - l_top), rounded once to bf16.  In fp32
        // first (the difference split exactly into hi + lo by Knuth's two-sum, exp(hi) (1 + lo), the sum in
        // order j = 0..k-1): within about a dozen fp32 ulps of the exact value, so where every p lies more
        // than kBf16Margin ulps from a bf16 rounding midpoint it rounds as the exact value does; otherwise
        // the warp takes fp64.
        float exf = 0.f;
        if (lane < k) {
            const float hi = my_l - top_l, bb = hi - my_l;
            const float lo = (my_l - (hi - bb)) + (-top_l - bb);      // my_l - top_l = hi + lo exactly
            exf = expf(hi) * (1.f + lo);
        }
        float denf = 0.f;
        for (int j = 0; j < k; ++j) denf += __shfl_sync(0xffffffffu, exf, j);
        const float pf = exf / denf;
        uint16_t pb = bf16_if_clear(pf);
        if (__any_sync(0xffffffffu, lane < k && pb == kBf16Unclear)) {
            double ex = 0.0;
            if (lane < k) ex = exp((double)my_l - (double)top_l);
            double den = 0.0;
            for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, ex, j);   // fixed order j = 0..k-1
            pb = double_to_bf16_bits(ex / den);
        }
        if (lane < k) {
            a.ids[(size_t)t * k + lane] = my_id;
            a.p[(size_t)t * k + lane] = pb;
            atomicAdd(a.hist + (size_t)(t / kTokBlock) * E + my_id, 1);
        }
        if (lane == 0 && a.w_s) {
            uint16_t ws = 0;
            if (a.has_shared) {
                // bf16(sigmoid(bf16(gamma))): fp32 first, fp64 near a rounding midpoint
                const float gb = bf16_bits_to_float(float_to_bf16_bits(a.gamma[t]));
                ws = bf16_if_clear(1.f / (1.f + expf(-gb)));
                if (ws == kBf16Unclear) ws = double_to_bf16_bits(1.0 / (1.0 + exp(-(double)gb)));
            }
            a.w_s[t] = ws;
        }
    }
}

// Exclusive prefix sum of a[0..n) in place, by one full warp; returns the total.
// Lane l scans a contiguous chunk, the chunk sums are scanned with shuffles.
__device__ int warp_exclusive_scan(int *a, int n)
{
    const int lane = threadIdx.x & 31;
    const int per = (n + 31) / 32;
    const int b = lane * per, e = min(n, b + per);
    int local = 0;
    for (int i = b; i < e; ++i) local += a[i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = b; i < e; ++i) {
        const int v = a[i];
        a[i] = run;
        run += v;
    }
    return __shfl_sync(0xffffffffu, incl, 31);
}

// Work lists of the expert kernels from the per-expert slot counts: expert e
// (in increasing id, the shared expert last as id E) contributes items of at most
// n tokens.  Decode GEMV list: n = 16.  GEMM lists (gate/up, down): an expert with at
// least kBigTok tokens gets items of kTileN1 / kTileN2 tokens for the tensor-memory
// GEMMs, placed first (nwork[3] / nwork[4] of them); the others get items of kSmallN
// tokens for the small-tile kernels, placed after.  Without small tiles (small == 0)
// every expert takes the first form.  Called by a whole block.
__device__ void build_work_lists(const int *s_cnt, int E, int T, int has_shared, int small, int32_t *nwork,
                                 WorkItem *work_dec, WorkItem *work_g1, WorkItem *work_g2, const int *max_items,
                                 int *status)
{
    // rows: 0 decode, 1 gate/up big, 2 down big, 3 gate/up small, 4 down small
    __shared__ int s_items[5][kMaxExperts + 2];
    const int tid = threadIdx.x;
    const int tile_n[5] = {kDecodeMaxTok, kTileN1, kTileN2, kSmallN, kSmallN};
    const int big_min = small ? kBigTok : 0;
    for (int w = 0; w < 5; ++w)
        for (int e = tid; e <= E; e += blockDim.x) {
            const int c = e < E ? s_cnt[e] : (has_shared ? T : 0);
            const bool take = w == 0 || (w < 3 ? c >= big_min : c < big_min);
            s_items[w][e] = take ? (c + tile_n[w] - 1) / tile_n[w] : 0;
        }
    __syncthreads();
    if (tid < 5 * 32) {
        const int w = tid >> 5;
        const int run = warp_exclusive_scan(s_items[w], E + 1);
        if ((tid & 31) == 0) s_items[w][E + 1] = run;
    }
    __syncthreads();
    if (tid == 0) {
        const int n1 = s_items[1][E + 1] + s_items[3][E + 1], n2 = s_items[2][E + 1] + s_items[4][E + 1];
        const bool bad = s_items[0][E + 1] > max_items[0] || n1 > max_items[1] || n2 > max_items[2];
        if (bad) record_status(status, MOE_ERR_DEVICE);   // counts inconsistent with T*k: build nothing
        nwork[0] = bad ? 0 : s_items[0][E + 1];
        nwork[1] = bad ? 0 : n1;
        nwork[2] = bad ? 0 : n2;
        nwork[3] = bad ? 0 : s_items[1][E + 1];
        nwork[4] = bad ? 0 : s_items[2][E + 1];
        s_items[0][E + 1] = bad ? -1 : s_items[0][E + 1];
    }
    __syncthreads();
    if (s_items[0][E + 1] < 0) return;
    WorkItem *lists[5] = {work_dec, work_g1, work_g2, work_g1, work_g2};
    for (int w = 0; w < 5; ++w) {
        const int base = w >= 3 ? s_items[w - 2][E + 1] : 0;   // small items after the big ones
        for (int e = tid; e <= E; e += blockDim.x) {
            const int c = e < E ? s_cnt[e] : (has_shared ? T : 0);
            int pos = base + s_items[w][e];
            const bool take = w == 0 || (w < 3 ? c >= big_min : c < big_min);
            if (!take) continue;
            for (int t0 = 0; t0 < c; t0 += tile_n[w]) {
                WorkItem it;
                it.expert = e;
                it.tok0 = t0;
                it.ntok = min(tile_n[w], c - t0);
                it.pad = 0;
                lists[w][pos++] = it;
            }
        }
    }
}

__global__ void __launch_bounds__(256) worklist_kernel(WorklistArgs a)
{
    __shared__ int s_cnt[kMaxExperts];
    if (threadIdx.x == 0) *a.status = 0;
    for (int i = threadIdx.x; i < a.nzero; i += blockDim.x) a.zero[i] = 0;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        int c = a.counts[e];
        if (c < 0 || c > a.T) {
            record_status(a.status, MOE_ERR_DEVICE);
            c = 0;
        }
        s_cnt[e] = c;
    }
    __syncthreads();
    build_work_lists(s_cnt, a.E, a.T, a.has_shared, a.small_tiles, a.nwork, a.work_dec, a.work_g1, a.work_g2, a.max_items,
                     a.status);
}

// Per-block histogram of the slots' expert ids (standalone permute call);
// clears the status word first (first kernel of that call).
__global__ void __launch_bounds__(1024) hist_kernel(HistArgs a)
{
    __shared__ int sh[kMaxExperts];
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) sh[e] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0;
    __syncthreads();
    const int f_begin = blockIdx.x * kTokBlock * a.k;
    const int f_end = min(a.T, (int)(blockIdx.x + 1) * kTokBlock) * a.k;
    for (int f = f_begin + threadIdx.x; f < f_end; f += blockDim.x) {
        const int e = a.ids[f];
        if (e >= 0 && e < a.E) atomicAdd(&sh[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) a.hist[(size_t)blockIdx.x * a.E + e] = sh[e];
}

// ---------------------------------------------------------------- permutation
//
// Block b owns the slots of tokens [128 b, 128 b + 128).  Every block sums the
// histogram column of each expert over all blocks (counts) and over the blocks
// before it (its base inside each expert's segment), scans counts into
// offsets, then scatters its own slots in increasing flat index: within a
// warp, lanes holding the same expert are ranked by __match_any_sync; across
// warps, by per-warp per-expert counts in shared memory.  Block 0 also writes
// counts/offsets and the work lists of the expert kernels.
__global__ void __launch_bounds__(1024) permute_kernel(PermuteArgs a)
{
    __shared__ int s_base[kMaxExperts];     // offsets[e] + slots of e in earlier blocks
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts + 1];
    __shared__ int s_wcnt[32][kMaxExperts]; // per-warp counts of the current chunk
    const int E = a.E, k = a.k, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int e = tid; e < E; e += blockDim.x) {
        int tot = 0, before = 0;
        for (int b = 0; b < a.nblk; ++b) {
            const int h = a.hist[(size_t)b * E + e];
            tot += h;
            if (b < (int)blockIdx.x) before += h;
        }
        s_cnt[e] = tot;
        s_base[e] = before;
    }
    __syncthreads();
    if (tid < 32) {
        for (int e = tid; e < E; e += 32) s_off[e] = s_cnt[e];
        __syncwarp();
        const int total = warp_exclusive_scan(s_off, E);
        if (tid == 0) s_off[E] = total;
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) s_base[e] += s_off[e];

    if (blockIdx.x == 0) {
        for (int e = tid; e < E; e += blockDim.x) a.counts[e] = s_cnt[e];
        for (int e = tid; e <= E; e += blockDim.x) a.offsets[e] = s_off[e];
        if (a.build_work)
            build_work_lists(s_cnt, E, a.T, a.has_shared, a.small_tiles, a.nwork, a.work_dec, a.work_g1, a.work_g2,
                             a.max_items,
                             a.status);
    }

    // stable scatter of this block's slots, 1024 at a time
    const int f_begin = blockIdx.x * kTokBlock * k;
    const int f_end = min(a.T, (int)(blockIdx.x + 1) * kTokBlock) * k;
    for (int c0 = f_begin; c0 < f_end; c0 += blockDim.x) {
        for (int i = tid; i < 32 * kMaxExperts; i += blockDim.x) (&s_wcnt[0][0])[i] = 0;
        __syncthreads();
        const int f = c0 + tid;
        const bool valid = f < f_end;
        int e = valid ? a.ids[f] : -1;
        if (valid && (e < 0 || e >= E)) {
            record_status(a.status, MOE_ERR_DEVICE);
            e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank_in_warp == 0) s_wcnt[warp][e] = __popc(peers);
        __syncthreads();
        if (e >= 0) {
            int before = 0;
            for (int w = 0; w < warp; ++w) before += s_wcnt[w][e];
            const int pos = s_base[e] + before + rank_in_warp;
            a.perm[pos] = f;
            a.inv_perm[f] = pos;
        }
        __syncthreads();
        for (int ee = tid; ee < E; ee += blockDim.x) {
            int tot = 0;
            for (int w = 0; w < 32; ++w) tot += s_wcnt[w][ee];
            s_base[ee] += tot;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- launchers

cudaError_t launch_route_gemv(const RouteArgs &a, cudaStream_t st)
{
    dim3 grid(a.n_expert_tiles + 1, (a.T + 7) / 8);
    route_gemv_kernel<<<grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_topk(const TopkArgs &a, cudaStream_t st)
{
    topk_kernel<<<(a.T + 7) / 8, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_hist(const HistArgs &a, cudaStream_t st)
{
    hist_kernel<<<a.nblk, 1024, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_worklist(const WorklistArgs &a, cudaStream_t st)
{
    worklist_kernel<<<1, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_permute(const PermuteArgs &a, cudaStream_t st)
{
    permute_kernel<<<a.nblk, 1024, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace qmoe
