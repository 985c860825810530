// Fused decode layer for T <= 16: one persistent launch after the router GEMV.
//
// The decode cost is the bytes of the selected experts (page "POC for qwen3.5 /
// qwen3.6 support optimized for AGX Orin", Phase 1-4: the batch-1 "gemv MoE
// path"; "both stacks are now weight-BW bound").  At T = 1 those are ~16 MB,
// a few microseconds of HBM time, so launch gaps and grid-wide barriers would
// dominate.  This kernel therefore keeps the whole expert stage in one grid of
// co-resident CTAs (cooperative launch) and replaces barriers by counters:
//   phase 0  every CTA stages x in shared memory, recomputes the top-k ids of
//            the <= 16 tokens from the fp32 logits (the same comparisons as the
//            top-k kernel) and builds the list of distinct experts (increasing
//            id, shared expert last) with their token columns; it also asks L2
//            to prefetch its share of the selected experts' down matrices.  The
//            pick weights and shared weight need fp64 (a long dependent chain
//            on this GPU), so only the first ceil(T/8) CTAs compute them, one
//            warp per token, publish them and skip phase 1; nothing but the
//            final combine waits for them;
//   phase 1  gate/up units (expert, 16 rows of I): split-K over the 8 warps,
//            fixed-order reduction, h = silu(g) * u stored as fp16; each unit
//            then increments its expert's counter;
//   phase 2  down units (expert, 128 rows of H), one per CTA, wait (one
//            polling thread, bounded, with backoff) for their expert's gate/up
//            units, write the raw expert output per slot; the last unit of each
//            128-row block (a per-block counter) combines that block for every
//            token in slot order and rounds once to bf16.
// The GEMV arithmetic (exact codes on mma.sync, per-group scale in fp32) is
// the one of the multi-kernel decode path; a token's result does not depend on
// the other tokens of the batch.  Counters are zeroed by the router kernel that
// precedes this launch on the stream.
#include <algorithm>

#include "kernels.cuh"

namespace qmoe {
namespace {

constexpr int kFThreads = 256;
constexpr int kCounterStride = 32;   // counters 128 bytes apart: pollers and writers do not share a line
constexpr int kMaxList = kMaxExperts + 1;

template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    if constexpr (F16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
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

template <bool F16>
__device__ __forceinline__ void nib8(uint32_t u, uint32_t *r)
{
    constexpr uint32_t base = F16 ? 0x64006400u : 0x43004300u;
    r[0] = (u & 0x000F000Fu) | base;
    r[1] = ((u >> 4) & 0x000F000Fu) | base;
    r[2] = ((u >> 8) & 0x000F000Fu) | base;
    r[3] = ((u >> 12) & 0x000F000Fu) | base;
}

__device__ __forceinline__ void permute_b(const uint4 &lo, const uint4 &hi, uint32_t *b)
{
    b[0] = prmt(lo.x, lo.z, 0x5410u);
    b[1] = prmt(lo.x, lo.z, 0x7632u);
    b[2] = prmt(lo.y, lo.w, 0x5410u);
    b[3] = prmt(lo.y, lo.w, 0x7632u);
    b[4] = prmt(hi.x, hi.z, 0x5410u);
    b[5] = prmt(hi.x, hi.z, 0x7632u);
    b[6] = prmt(hi.y, hi.w, 0x5410u);
    b[7] = prmt(hi.y, hi.w, 0x7632u);
}

template <bool F16>
__device__ __forceinline__ void group_mma(uint2 c_lo, uint2 c_hi, const uint32_t *bp, float (&dq)[4],
                                          float (&dx)[4], bool do_ones)
{
    constexpr uint32_t ones = F16 ? 0x3C003C00u : 0x3F803F80u;
    uint32_t ra[8], rb[8];
    nib8<F16>(c_lo.x, ra);
    nib8<F16>(c_lo.y, ra + 4);
    nib8<F16>(c_hi.x, rb);
    nib8<F16>(c_hi.y, rb + 4);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        mma16816<F16>(dq, ra[2 * m], rb[2 * m], ra[2 * m + 1], rb[2 * m + 1], bp[2 * m], bp[2 * m + 1]);
        if (do_ones) mma16816<F16>(dx, ones, ones, ones, ones, bp[2 * m], bp[2 * m + 1]);
    }
}

__device__ __forceinline__ uint32_t logit_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) == 0) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int ld_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

struct Smem {
    int ids[kDecodeMaxTok][kMaxTopK];
    float lg[kDecodeMaxTok][kMaxTopK];     // fp32 logit of each pick
    float p[kDecodeMaxTok][kMaxTopK];
    uint16_t pbits[kDecodeMaxTok][kMaxTopK];
    float ws[kDecodeMaxTok];
    uint16_t wsbits[kDecodeMaxTok];
    int flag[kMaxExperts];
    int list[kMaxList];
    int ncols[kMaxList];
    int cols[kMaxList][kDecodeMaxTok];     // slot index f of each column
    int nlist;
    float red[8][2][16][kDecodeMaxTok];    // split-K partials of a gate/up unit
};

__device__ __forceinline__ const uint8_t *codes_of(const QMatDev &m, int e, int rows, int cols)
{
    return m.codes + (size_t)e * rows * (cols / 2);
}
__device__ __forceinline__ size_t sb_off(int e, int rows, int cols) { return (size_t)e * rows * (cols / kGroup); }

// ------------------------------------------------------------------ kernel
template <int NT, bool XS>
__global__ void __launch_bounds__(kFThreads, 2) decode_fused_kernel(FusedDecodeArgs a)
{
    __shared__ Smem S;
    extern __shared__ uint4 s_x[];         // XS: x rows [T][H/8 + 1] (one uint4 of padding per row)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k;
    const int G = H / kGroup, GI = I / kGroup, rowu4 = H / 8 + 1;
    // CTAs [0, npc) compute the fp64 pick weights (one warp per token) and skip phase 1
    const int npc = a.ids_in ? 0 : (T + 7) / 8;
    if (XS)
        for (int i = tid; i < T * (H / 8); i += kFThreads) {
            const int tt = i / (H / 8), col = i - tt * (H / 8);
            s_x[tt * rowu4 + col] = __ldg(reinterpret_cast<const uint4 *>(a.x + (size_t)tt * H) + col);
        }

    // ---------------------------------------------------------------- phase 0: routing
    if (a.ids_in) {
        // routing given by the caller (the staged expert-FFN entry point)
        for (int i = tid; i < T * k; i += kFThreads) {
            const int tt = i / k, j = i - tt * k;
            int e = a.ids_in[i];
            if (e < 0 || e >= E) {
                record_status(a.status, MOE_ERR_DEVICE);
                e = 0;
            }
            S.ids[tt][j] = e;
            S.pbits[tt][j] = a.p_in[i];
            S.p[tt][j] = bf16_bits_to_float(a.p_in[i]);
        }
        for (int tt = tid; tt < T; tt += kFThreads) {
            const uint16_t wsb = (a.has_shared && a.ws_in) ? a.ws_in[tt] : (uint16_t)0;
            S.wsbits[tt] = wsb;
            S.ws[tt] = bf16_bits_to_float(wsb);
        }
    } else
    for (int tt = warp; tt < T; tt += 8) {
        const float *lrow = a.logits + (size_t)tt * E;
        uint32_t key[kMaxExperts / 32];
        float val[kMaxExperts / 32];
#pragma unroll
        for (int r = 0; r < kMaxExperts / 32; ++r) {
            const int e = lane + 32 * r;
            val[r] = e < E ? lrow[e] : 0.f;
            key[r] = e < E ? logit_key(val[r]) : 0u;
        }
        unsigned taken = 0;
        float top_l = 0.f, my_l = 0.f;
        int my_id = -1;
        for (int j = 0; j < k; ++j) {
            unsigned long long best = 0;
#pragma unroll
            for (int r = 0; r < kMaxExperts / 32; ++r) {
                const int e = lane + 32 * r;
                if (e < E && !(taken & (1u << r))) {
                    const unsigned long long c = ((unsigned long long)key[r] << 32) | (unsigned)(0xFFFF - e);
                    best = c > best ? c : best;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
                best = other > best ? other : best;
            }
            const int id = 0xFFFF - (int)(best & 0xFFFFu);
            if ((id & 31) == lane) taken |= 1u << (id >> 5);
            float v = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxExperts / 32; ++r)
                if ((id >> 5) == r) v = val[r];
            v = __shfl_sync(0xffffffffu, v, id & 31);
            if (j == 0) top_l = v;
            if (lane == j) { my_id = id; my_l = v; }
        }
        (void)top_l;
        if (lane < k) {
            S.ids[tt][lane] = my_id;
            S.lg[tt][lane] = my_l;
        }
    }
    __syncthreads();
    if (blockIdx.x == 0 && !a.ids_in && a.ids_out)
        for (int i = tid; i < T * k; i += kFThreads) a.ids_out[i] = S.ids[i / k][i % k];
    if ((int)blockIdx.x < npc) {
        // pick weights p = exp(l - l_top) / sum over the picks and w_s = sigmoid(bf16(gamma)),
        // in fp64 with one rounding to bf16; published for the combining CTAs
        const int tt = blockIdx.x * 8 + warp;
        if (tt < T) {
            double ex = 0.0;
            if (lane < k) ex = exp((double)S.lg[tt][lane] - (double)S.lg[tt][0]);
            double den = 0.0;
            for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, ex, j);
            if (lane < k) {
                const uint16_t pb = double_to_bf16_bits(ex / den);
                a.p_glob[tt * k + lane] = pb;
                if (a.p_out) a.p_out[tt * k + lane] = pb;
            }
            if (lane == 0) {
                uint16_t wsb = 0;
                if (a.has_shared) {
                    const float gb = bf16_bits_to_float(float_to_bf16_bits(a.gamma[tt]));
                    wsb = double_to_bf16_bits(1.0 / (1.0 + exp(-(double)gb)));
                }
                a.ws_glob[tt] = wsb;
                if (a.ws_out) a.ws_out[tt] = wsb;
            }
        }
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            atomicAdd(a.cnt_pick, 1);
        }
    }
    // distinct experts in increasing id, then the shared expert
    for (int e = tid; e < E; e += kFThreads) {
        int used = 0;
        for (int i = 0; i < T * k; ++i) used |= S.ids[i / k][i % k] == e;
        S.flag[e] = used;
    }
    __syncthreads();
    if (warp == 0) {
        const int per = (E + 31) / 32, b0 = lane * per, b1 = min(E, b0 + per);
        int local = 0;
        for (int e = b0; e < b1; ++e) local += S.flag[e];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int pos = incl - local;
        for (int e = b0; e < b1; ++e)
            if (S.flag[e]) S.list[pos++] = e;
        if (lane == 31) {
            S.nlist = incl + (a.has_shared ? 1 : 0);
            if (a.has_shared) S.list[incl] = E;
        }
    }
    __syncthreads();
    const int D = S.nlist;
    for (int d = tid; d < D; d += kFThreads) {
        const int e = S.list[d];
        int n = 0;
        if (e == E) {
            for (int tt = 0; tt < T; ++tt) S.cols[d][n++] = T * k + tt;
        } else {
            for (int tt = 0; tt < T; ++tt)
                for (int j = 0; j < k; ++j)
                    if (S.ids[tt][j] == e) {
                        if (n < kDecodeMaxTok) S.cols[d][n++] = tt * k + j;
                        else record_status(a.status, MOE_ERR_DEVICE);   // an id repeated within a token
                    }
        }
        S.ncols[d] = n;
    }
    __syncthreads();

    // L2 prefetch of the selected experts' down matrices (codes in 64 KB pieces, scales, biases)
    {
        const size_t dcode = (size_t)H * (I / 2), dsb = (size_t)H * GI * 2;
        const int pieces = (int)((dcode + 65535) / 65536) + 2;
        for (int q = blockIdx.x + tid * gridDim.x; q < D * pieces; q += gridDim.x * kFThreads) {   // one piece per CTA first
            const int d = q / pieces, piece = q - d * pieces;
            const int e = S.list[d];
            const QMatDev &m = e == E ? a.s_down : a.down;
            const int ee = e == E ? 0 : e;
            if (piece < pieces - 2) {
                const size_t off = (size_t)piece * 65536;
                const uint32_t bytes = (uint32_t)(dcode - off < 65536 ? dcode - off : 65536);
                prefetch_l2(codes_of(m, ee, H, I) + off, bytes);
            } else {
                const uint16_t *p = piece == pieces - 2 ? m.scales : m.biases;
                prefetch_l2(p + sb_off(ee, H, I), (uint32_t)dsb);
            }
        }
    }

    // ---------------------------------------------------------------- phase 1: gate/up units
    const int rb_i = I / 16;
    const int U1 = D * rb_i;
    const int p1_cta = (int)blockIdx.x - npc, p1_grid = (int)gridDim.x - npc;
    for (int u = p1_cta; p1_cta >= 0 && u < U1; u += p1_grid) {
        const int d = u / rb_i, rb = u - d * rb_i;
        const int e = S.list[d];
        const bool shr = e == E;
        const int ee = shr ? 0 : e;
        const QMatDev &mg = shr ? a.s_gate : a.gate, &mu = shr ? a.s_up : a.up;
        const uint8_t *cg = codes_of(mg, ee, I, H), *cu = codes_of(mu, ee, I, H);
        const size_t so = sb_off(ee, I, H);
        const int r0 = rb * 16 + g, r1 = r0 + 8;
        const int gbeg = (warp * G) / 8, gend = ((warp + 1) * G) / 8;
        const int ncol = S.ncols[d];
        int xrow[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int c = j * 8 + g;
            const int f = c < ncol ? S.cols[d][c] : -1;
            xrow[j] = f < 0 ? -1 : (f >= T * k ? f - T * k : f / k);
        }
        float acc_g[NT][4], acc_u[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc_g[j][q] = acc_u[j][q] = 0.f;
        constexpr int GB = 4;
        for (int gb = gbeg; gb < gend; gb += GB) {
            uint2 cg0[GB], cg1[GB], cu0[GB], cu1[GB];
            uint16_t sg[GB][2], bg[GB][2], su[GB][2], bu[GB][2];
#pragma unroll
            for (int i = 0; i < GB; ++i) {
                const int grp = gb + i;
                if (grp < gend) {
                    const size_t co = (size_t)grp * 32 + 8 * t4;
                    cg0[i] = __ldg(reinterpret_cast<const uint2 *>(cg + (size_t)r0 * (H / 2) + co));
                    cg1[i] = __ldg(reinterpret_cast<const uint2 *>(cg + (size_t)r1 * (H / 2) + co));
                    cu0[i] = __ldg(reinterpret_cast<const uint2 *>(cu + (size_t)r0 * (H / 2) + co));
                    cu1[i] = __ldg(reinterpret_cast<const uint2 *>(cu + (size_t)r1 * (H / 2) + co));
                    sg[i][0] = __ldg(mg.scales + so + (size_t)r0 * G + grp);
                    sg[i][1] = __ldg(mg.scales + so + (size_t)r1 * G + grp);
                    bg[i][0] = __ldg(mg.biases + so + (size_t)r0 * G + grp);
                    bg[i][1] = __ldg(mg.biases + so + (size_t)r1 * G + grp);
                    su[i][0] = __ldg(mu.scales + so + (size_t)r0 * G + grp);
                    su[i][1] = __ldg(mu.scales + so + (size_t)r1 * G + grp);
                    bu[i][0] = __ldg(mu.biases + so + (size_t)r0 * G + grp);
                    bu[i][1] = __ldg(mu.biases + so + (size_t)r1 * G + grp);
                }
            }
#pragma unroll
            for (int i = 0; i < GB; ++i) {
                const int grp = gb + i;
                if (grp >= gend) break;
                const float s_g0 = bf16_bits_to_float(sg[i][0]), s_g1 = bf16_bits_to_float(sg[i][1]);
                const float s_u0 = bf16_bits_to_float(su[i][0]), s_u1 = bf16_bits_to_float(su[i][1]);
                const float c_g0 = fmaf(-128.f, s_g0, bf16_bits_to_float(bg[i][0]));
                const float c_g1 = fmaf(-128.f, s_g1, bf16_bits_to_float(bg[i][1]));
                const float c_u0 = fmaf(-128.f, s_u0, bf16_bits_to_float(bu[i][0]));
                const float c_u1 = fmaf(-128.f, s_u1, bf16_bits_to_float(bu[i][1]));
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    uint32_t bp[8];
                    if (xrow[j] >= 0) {
                        if (XS) {
                            const uint4 *xr = s_x + xrow[j] * rowu4 + grp * 8 + 2 * t4;
                            permute_b(xr[0], xr[1], bp);
                        } else {
                            const uint4 *xr =
                                reinterpret_cast<const uint4 *>(a.x + (size_t)xrow[j] * H) + grp * 8 + 2 * t4;
                            permute_b(__ldg(xr), __ldg(xr + 1), bp);
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; ++q) bp[q] = 0;
                    }
                    float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f}, dx[4] = {0.f, 0.f, 0.f, 0.f};
                    group_mma<false>(cg0[i], cg1[i], bp, dg, dx, true);
                    group_mma<false>(cu0[i], cu1[i], bp, du, dx, false);
                    acc_g[j][0] = fmaf(s_g0, dg[0], fmaf(c_g0, dx[0], acc_g[j][0]));
                    acc_g[j][1] = fmaf(s_g0, dg[1], fmaf(c_g0, dx[1], acc_g[j][1]));
                    acc_g[j][2] = fmaf(s_g1, dg[2], fmaf(c_g1, dx[2], acc_g[j][2]));
                    acc_g[j][3] = fmaf(s_g1, dg[3], fmaf(c_g1, dx[3], acc_g[j][3]));
                    acc_u[j][0] = fmaf(s_u0, du[0], fmaf(c_u0, dx[0], acc_u[j][0]));
                    acc_u[j][1] = fmaf(s_u0, du[1], fmaf(c_u0, dx[1], acc_u[j][1]));
                    acc_u[j][2] = fmaf(s_u1, du[2], fmaf(c_u1, dx[2], acc_u[j][2]));
                    acc_u[j][3] = fmaf(s_u1, du[3], fmaf(c_u1, dx[3], acc_u[j][3]));
                }
            }
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int c0 = j * 8 + 2 * t4;
            S.red[warp][0][g][c0] = acc_g[j][0];
            S.red[warp][0][g][c0 + 1] = acc_g[j][1];
            S.red[warp][0][g + 8][c0] = acc_g[j][2];
            S.red[warp][0][g + 8][c0 + 1] = acc_g[j][3];
            S.red[warp][1][g][c0] = acc_u[j][0];
            S.red[warp][1][g][c0 + 1] = acc_u[j][1];
            S.red[warp][1][g + 8][c0] = acc_u[j][2];
            S.red[warp][1][g + 8][c0 + 1] = acc_u[j][3];
        }
        __syncthreads();
        {
            const int row = tid & 15, c = tid >> 4;   // 256 threads = 16 rows x 16 columns
            if (c < ncol && c < NT * 8) {
                float gs = 0.f, us = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    gs += S.red[w][0][row][c];
                    us += S.red[w][1][row][c];
                }
                const float hv = gs / (1.f + __expf(-gs)) * us;
                a.h[(size_t)S.cols[d][c] * I + rb * 16 + row] = __half_as_ushort(__float2half_rn(hv));
            }
        }
        __syncthreads();
        if (tid == 0) {
            __threadfence();                 // cumulative: every h store of this unit is visible first
            atomicAdd(a.cnt_expert + d * kCounterStride, 1);
        }
    }

    // ---------------------------------------------------------------- phase 2: down units + combine
    // Unit = (expert d, 128-row block of H); warp w owns rows 16 w .. 16 w + 15 of it.
    // Thread 0 alone waits (with backoff) for the expert's gate/up units.
    const int rb_h = (H + 127) / 128;
    const int U2 = D * rb_h;
    __shared__ int s_ready;
    for (int v = blockIdx.x; v < U2; v += gridDim.x) {
        const int d = v / rb_h, rb = v - d * rb_h;
        const int e = S.list[d];
        const bool shr = e == E;
        const int ee = shr ? 0 : e;
        const QMatDev &md = shr ? a.s_down : a.down;
        const uint8_t *cd = codes_of(md, ee, H, I);
        const size_t so = sb_off(ee, H, I);
        const int rbase = rb * 128 + warp * 16;
        const bool wactive = rbase < H;
        const int r0 = min(rbase + g, H - 1), r1 = min(rbase + g + 8, H - 1);
        const int ncol = S.ncols[d];
        constexpr int GBD = 8;
        float acc[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;
        for (int gb = 0; gb < GI; gb += GBD) {
            uint2 c0[GBD], c1[GBD];
            uint16_t sv[GBD][2], bv[GBD][2];
#pragma unroll
            for (int i = 0; i < GBD; ++i) {
                const int grp = gb + i;
                if (grp < GI) {
                    const size_t co = (size_t)grp * 32 + 8 * t4;
                    c0[i] = __ldg(reinterpret_cast<const uint2 *>(cd + (size_t)r0 * (I / 2) + co));
                    c1[i] = __ldg(reinterpret_cast<const uint2 *>(cd + (size_t)r1 * (I / 2) + co));
                    sv[i][0] = __ldg(md.scales + so + (size_t)r0 * GI + grp);
                    sv[i][1] = __ldg(md.scales + so + (size_t)r1 * GI + grp);
                    bv[i][0] = __ldg(md.biases + so + (size_t)r0 * GI + grp);
                    bv[i][1] = __ldg(md.biases + so + (size_t)r1 * GI + grp);
                }
            }
            if (gb == 0) {
                // the codes above are in flight; now wait for this expert's h
                if (tid == 0) {
                    const int *cnt = a.cnt_expert + d * kCounterStride;
                    long long n = 0;
                    unsigned ns = 64;
                    while (ld_acquire(cnt) < rb_i && n <= a.wait_limit) {
                        ++n;
                        __nanosleep(ns);
                        ns = ns < 1024 ? ns * 2 : 1024;
                    }
                    const int ok = n <= a.wait_limit;
                    if (!ok) record_status(a.status, MOE_ERR_TIMEOUT);
                    s_ready = ok;
                }
                __syncthreads();
                if (!s_ready) break;
            }
#pragma unroll
            for (int i = 0; i < GBD; ++i) {
                const int grp = gb + i;
                if (grp >= GI) break;
                const float s0 = bf16_bits_to_float(sv[i][0]), s1 = bf16_bits_to_float(sv[i][1]);
                const float k0 = fmaf(-1024.f, s0, bf16_bits_to_float(bv[i][0]));
                const float k1 = fmaf(-1024.f, s1, bf16_bits_to_float(bv[i][1]));
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int c = j * 8 + g;
                    const int f = c < ncol ? S.cols[d][c] : -1;
                    uint32_t bp[8];
                    if (f >= 0) {
                        const uint4 *hr = reinterpret_cast<const uint4 *>(a.h + (size_t)f * I) + grp * 8 + 2 * t4;
                        permute_b(__ldcg(hr), __ldcg(hr + 1), bp);
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; ++q) bp[q] = 0;
                    }
                    float dd[4] = {0.f, 0.f, 0.f, 0.f}, dx[4] = {0.f, 0.f, 0.f, 0.f};
                    group_mma<true>(c0[i], c1[i], bp, dd, dx, true);
                    acc[j][0] = fmaf(s0, dd[0], fmaf(k0, dx[0], acc[j][0]));
                    acc[j][1] = fmaf(s0, dd[1], fmaf(k0, dx[1], acc[j][1]));
                    acc[j][2] = fmaf(s1, dd[2], fmaf(k1, dx[2], acc[j][2]));
                    acc[j][3] = fmaf(s1, dd[3], fmaf(k1, dx[3], acc[j][3]));
                }
            }
        }
        if (!s_ready) {
            __syncthreads();
            continue;
        }
        if (wactive) {
            const int w0 = rbase + g, w1 = w0 + 8;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int cA = j * 8 + 2 * t4, cB = cA + 1;
                if (cA < ncol) {
                    const int f = S.cols[d][cA];
                    a.yslot[(size_t)f * H + w0] = acc[j][0];
                    a.yslot[(size_t)f * H + w1] = acc[j][2];
                }
                if (cB < ncol) {
                    const int f = S.cols[d][cB];
                    a.yslot[(size_t)f * H + w0] = acc[j][1];
                    a.yslot[(size_t)f * H + w1] = acc[j][3];
                }
            }
        }
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            s_ready = atomicAdd(a.cnt_rows + rb * kCounterStride, 1) == D - 1 ? 2 : 1;
        }
        __syncthreads();
        if (s_ready == 2 && !a.ids_in) {
            // wait (bounded) for the published pick weights, then take them into shared memory
            if (tid == 0) {
                long long n = 0;
                unsigned ns = 64;
                while (ld_acquire(a.cnt_pick) < npc && n <= a.wait_limit) {
                    ++n;
                    __nanosleep(ns);
                    ns = ns < 1024 ? ns * 2 : 1024;
                }
                if (n > a.wait_limit) {
                    record_status(a.status, MOE_ERR_TIMEOUT);
                    s_ready = 1;
                }
            }
            __syncthreads();
            if (s_ready == 2) {
                for (int i = tid; i < T * k; i += kFThreads) S.p[i / k][i % k] = bf16_bits_to_float(__ldcg(a.p_glob + i));
                for (int tt = tid; tt < T; tt += kFThreads) S.ws[tt] = bf16_bits_to_float(__ldcg(a.ws_glob + tt));
            }
            __syncthreads();
        }
        if (s_ready == 2) {
            __threadfence();
            // last unit of this row block: y = bf16(sum_j p_j y_slot[t*k+j] + w_s y_slot[T*k+t]), slot order
            const int nrow = min(128, H - rb * 128);
            for (int q = tid; q < nrow * T; q += kFThreads) {
                const int tt = q / nrow, row = rb * 128 + (q - tt * nrow);
                float s = 0.f;
                for (int j = 0; j < k; ++j) s = fmaf(S.p[tt][j], __ldcg(a.yslot + ((size_t)tt * k + j) * H + row), s);
                if (a.has_shared) s = fmaf(S.ws[tt], __ldcg(a.yslot + ((size_t)T * k + tt) * H + row), s);
                if (a.y)
                    a.y[(size_t)tt * H + row] = float_to_bf16_bits(s);
                else
                    a.acc[(size_t)tt * H + row] += s;
            }
        }
        __syncthreads();
    }
}

struct Occupancy {
    int device = -1;
    size_t smem = 0;
    int sms = 0;
    int per_sm = 0;
};

}  // namespace

cudaError_t launch_decode_fused(const FusedDecodeArgs &a, cudaStream_t st)
{
    static Occupancy occ[16][4];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int nt = a.T > 8 ? 1 : 0;
    const size_t xs_bytes = (size_t)a.T * (a.H / 8 + 1) * 16;
    const bool xs = xs_bytes <= 100 * 1024;
    const int variant = nt * 2 + (xs ? 1 : 0);
    auto kern = variant == 0 ? decode_fused_kernel<1, false>
              : variant == 1 ? decode_fused_kernel<1, true>
              : variant == 2 ? decode_fused_kernel<2, false>
                             : decode_fused_kernel<2, true>;
    const size_t smem = xs ? xs_bytes : 0;
    Occupancy &o = occ[dev & 15][variant];
    if (o.device != dev || o.smem != smem) {
        if ((e = cudaDeviceGetAttribute(&o.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(100 * 1024 + 1024))) !=
            cudaSuccess)
            return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o.per_sm, kern, kFThreads, smem)) != cudaSuccess)
            return e;
        o.device = dev;
        o.smem = smem;
    }
    if (o.per_sm < 1) return cudaErrorInvalidConfiguration;
    const int grid = o.sms * std::min(2, o.per_sm);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace qmoe
