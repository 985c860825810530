// Decode path: weight-streaming dequant-GEMV over the selected experts.
//
// Meant for small token counts (the "gemv MoE path" at batch size 1 of the page
// "POC for qwen3.5 / qwen3.6 support optimized for AGX Orin", Phase 1-4): the
// cost is the bytes of the experts the batch selected, each streamed from HBM
// exactly once, whatever number of the batch's tokens picked it.
//
// Arithmetic.  A weight of group g of a row is w = s_g * q + b_g (MLX affine,
// 4-bit codes, group 64).  Over one group of 64 inputs
//     sum_j w_j x_j = s_g * sum_j (128 + q_j) x_j + (b_g - 128 s_g) * sum_j x_j.
// 128 + q is exact in bf16 (OR of the nibble into the mantissa of 128.0), and
// the products with a bf16 x are exact, so the two sums are computed on the
// tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate): one MMA chain
// with the codes as A, and one with an all-ones A that yields sum_j x_j.  The
// per-group scale and bias are then applied in fp32 per row.  The down
// projection works the same way in fp16: 1024 + q is exact in fp16 and the
// intermediate h is stored as fp16.  Nothing of a weight is rounded; the only
// rounding before fp32 accumulation is the fp16 storage of h (11 significant
// bits: bf16's 8 would put the layer output outside the parity tolerance).
//
// Fragment layout.  Thread (g = lane/4, t = lane%4) loads the 16 codes of
// inputs 16t..16t+15 of rows g and g+8 of a group (8 bytes of 4-bit codes, 16
// bytes of 8-bit codes).  Eight codes split into four bf16x2 registers holding
// elements (0,4) (1,5) (2,6) (3,7); MMA m of the group's four takes registers
// 2m, 2m+1.  The MMA's k order is therefore a permutation of the group's inputs;
// the B fragment (x or h) is permuted the same way with byte permutes, so each
// product still pairs w_j with x_j.  Every output element is one column of the
// MMA and never mixes tokens, so a token's result does not depend on the batch
// it is in.
//
// 8-bit codes (the "8-bit experts" slice of the page on Qwen3.6-35B-A3B on the
// native Metal engine: the same affine rule with q in [0, 255]).  1024 + q is
// still exact in fp16, so the down projection only swaps the code expansion.
// In bf16 only 128 + n with n < 128 is exact, so the gate/up projection splits
// q = 16 qh + ql into nibbles and runs two code chains:
//     sum_j q_j x_j = 16 sum_j (128 + qh_j) x_j + sum_j (128 + ql_j) x_j - 2176 sum_j x_j,
// with the 2176 folded into the bias term as for the 4-bit codes.
#include <type_traits>

#include "kernels.cuh"

namespace qmoe {
namespace {

// D += A B, m16n8k16, fp32 accumulate; F16 selects fp16 operands, else bf16.
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

// 8 nibbles -> four 16-bit pairs of (OFF + q), elements (0,4), (1,5), (2,6), (3,7).
// bf16: OR into the mantissa of 128.0 (0x4300) gives 128 + q exactly; fp16: OR
// into the mantissa of 1024.0 (0x6400) gives 1024 + q exactly.
template <bool F16>
__device__ __forceinline__ void nib8(uint32_t u, uint32_t *r)
{
    constexpr uint32_t base = F16 ? 0x64006400u : 0x43004300u;
    r[0] = (u & 0x000F000Fu) | base;
    r[1] = ((u >> 4) & 0x000F000Fu) | base;
    r[2] = ((u >> 8) & 0x000F000Fu) | base;
    r[3] = ((u >> 12) & 0x000F000Fu) | base;
}

// Byte pairs (0,4), (1,5), (2,6), (3,7) of 8 byte codes (u0: codes 0-3, u1: codes 4-7), each pair in
// bytes 0 and 2 of a word (bytes 1 and 3 are copies, masked off by the callers).
__device__ __forceinline__ void byte_pairs(uint32_t u0, uint32_t u1, uint32_t *t)
{
    t[0] = prmt(u0, u1, 0x4400u);
    t[1] = prmt(u0, u1, 0x5511u);
    t[2] = prmt(u0, u1, 0x6622u);
    t[3] = prmt(u0, u1, 0x7733u);
}

// 16 byte codes -> eight fp16x2 of 1024 + q (exact), elements (0,4) (1,5) (2,6) (3,7) (8,12) ... (11,15).
__device__ __forceinline__ void byte16_f16(uint4 c, uint32_t *r)
{
    uint32_t t[8];
    byte_pairs(c.x, c.y, t);
    byte_pairs(c.z, c.w, t + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = (t[i] & 0x00FF00FFu) | 0x64006400u;
}

// 16 byte codes -> eight bf16x2 of 128 + ql (lo) and eight of 128 + qh (hi), q = 16 qh + ql, in the
// element order of byte16_f16.
__device__ __forceinline__ void byte16_nibbles(uint4 c, uint32_t *lo, uint32_t *hi)
{
    uint32_t t[8];
    byte_pairs(c.x, c.y, t);
    byte_pairs(c.z, c.w, t + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        lo[i] = (t[i] & 0x000F000Fu) | 0x43004300u;
        hi[i] = ((t[i] >> 4) & 0x000F000Fu) | 0x43004300u;
    }
}

// 16 consecutive bf16 (two uint4) -> eight bf16x2 in the codes' element order.
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

// One group (64 inputs) of a 16-row block against one n8 tile of B:
// codes u64 of rows g / g+8, B registers bp[8]; accumulates the code chain
// sum (OFF + q) b and, with do_ones, the ones chain sum b over the group.
// The same with the code registers ra (row g) and rb (row g+8) already expanded.
template <bool F16>
__device__ __forceinline__ void group_mma_regs(const uint32_t *ra, const uint32_t *rb, const uint32_t *bp,
                                               float (&dq)[4], float (&dx)[4], bool do_ones)
{
    constexpr uint32_t ones = F16 ? 0x3C003C00u : 0x3F803F80u;   // {1, 1}
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        mma16816<F16>(dq, ra[2 * m], rb[2 * m], ra[2 * m + 1], rb[2 * m + 1], bp[2 * m], bp[2 * m + 1]);
        if (do_ones) mma16816<F16>(dx, ones, ones, ones, ones, bp[2 * m], bp[2 * m + 1]);
    }
}

template <bool F16>
__device__ __forceinline__ void group_mma(uint2 c_lo, uint2 c_hi, const uint32_t *bp, float (&dq)[4],
                                          float (&dx)[4], bool do_ones)
{
    uint32_t ra[8], rb[8];
    nib8<F16>(c_lo.x, ra);
    nib8<F16>(c_lo.y, ra + 4);
    nib8<F16>(c_hi.x, rb);
    nib8<F16>(c_hi.y, rb + 4);
    group_mma_regs<F16>(ra, rb, bp, dq, dx, do_ones);
}

// Down projection, 8-bit codes: chain of 1024 + q (fp16) and, with do_ones, the ones chain.
__device__ __forceinline__ void group_mma(uint4 c_lo, uint4 c_hi, const uint32_t *bp, float (&dq)[4],
                                          float (&dx)[4], bool do_ones)
{
    uint32_t ra[8], rb[8];
    byte16_f16(c_lo, ra);
    byte16_f16(c_hi, rb);
    group_mma_regs<true>(ra, rb, bp, dq, dx, do_ones);
}

// Gate/up projection, 8-bit codes (bf16): dq = 16 sum (128 + qh) b + sum (128 + ql) b = sum (2176 + q) b.
__device__ __forceinline__ void group_mma_bf16_b8(uint4 c_lo, uint4 c_hi, const uint32_t *bp, float (&dq)[4],
                                                  float (&dx)[4], bool do_ones)
{
    uint32_t la[8], ha[8], lb[8], hb[8];
    byte16_nibbles(c_lo, la, ha);
    byte16_nibbles(c_hi, lb, hb);
    float dh[4] = {0.f, 0.f, 0.f, 0.f};
    group_mma_regs<false>(la, lb, bp, dq, dx, do_ones);
    group_mma_regs<false>(ha, hb, bp, dh, dx, false);
#pragma unroll
    for (int i = 0; i < 4; ++i) dq[i] = fmaf(16.f, dh[i], dq[i]);
}

struct ExpertView {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint16_t *biases;
};

__device__ __forceinline__ ExpertView expert_view(const QMatDev &m, int e, int rows, int cols, int bits)
{
    ExpertView v;
    const size_t eo = (size_t)e * rows;
    v.codes = m.codes + eo * ((size_t)cols * bits / 8);
    v.scales = m.scales + eo * (cols / kGroup);
    v.biases = m.biases + eo * (cols / kGroup);
    return v;
}

// Columns (tokens) of a work item: token index and slot index f.
__device__ __forceinline__ void item_columns(const ExpertArgs &a, const WorkItem &it, int *s_tok, int *s_slot)
{
    const int c = threadIdx.x;
    if (c < kDecodeMaxTok) {
        int t = -1, f = -1;
        if (c < it.ntok) {
            if (it.expert == a.E) {
                t = it.tok0 + c;
                f = a.T * a.k + t;
            } else {
                const int pos = __ldg(a.offsets + it.expert) + it.tok0 + c;
                f = (pos >= 0 && pos < a.T * a.k) ? __ldg(a.perm + pos) : -1;
                if (f < 0 || f >= a.T * a.k) {      // offsets/perm inconsistent with the work list
                    record_status(a.status, MOE_ERR_DEVICE);
                    f = -1;
                }
                t = f < 0 ? -1 : f / a.k;
            }
        }
        s_tok[c] = t;
        s_slot[c] = f;
    }
}

// ------------------------------------------------------------ gate/up + SwiGLU
//
// grid (I/16, max items); 256 threads.  Block (rb, item) computes rows
// [16 rb, 16 rb + 16) of gate and up for the item's <= 16 tokens; warp w takes
// an eighth of the hidden groups and the eighths are added in warp order (the
// same split and order as the fused decode kernel, so both give the same bits).
// BITS: expert code width (4 or 8).
template <int NT, int BITS>
__global__ void __launch_bounds__(256) decode_gateup_kernel(ExpertArgs a)
{
    extern __shared__ uint4 s_x[];                 // [NT*8][H/8 + 1] (one uint4 of padding per row)
    __shared__ float s_red[8][2][16][NT * 8];      // [warp][gate/up][row][col]
    __shared__ int s_tok[kDecodeMaxTok], s_slot[kDecodeMaxTok], s_e[kDecodeMaxTok];
    if ((int)blockIdx.y >= __ldg(a.nwork + 0)) return;
    const WorkItem it = a.work[blockIdx.y];
    const int H = a.H, I = a.I, G = H / kGroup, rowu4 = H / 8 + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const bool is_shared = it.expert == a.E;

    item_columns(a, it, s_tok, s_slot);
    __syncthreads();
    for (int idx = threadIdx.x; idx < NT * 8 * (H / 8); idx += blockDim.x) {
        const int c = idx / (H / 8), col = idx - c * (H / 8);
        const int tok = c < kDecodeMaxTok ? s_tok[c] : -1;
        s_x[c * rowu4 + col] = tok >= 0 ? __ldg(reinterpret_cast<const uint4 *>(a.x + (size_t)tok * H) + col)
                                        : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    // e of each column's token (2^e <= max |x| < 2^(e + 1)): h is stored as fp16 h 2^-2e, which stays
    // inside the fp16 range whatever the size of x; the down kernel undoes the scale (exact)
    for (int c = warp; c < NT * 8 && c < kDecodeMaxTok; c += 8) {
        uint32_t mx = 0;
        for (int col = lane; col < H / 8; col += 32) {
            const uint4 v = s_x[c * rowu4 + col];
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) mx = max(mx, max(w4[q] & 0x7FFFu, (w4[q] >> 16) & 0x7FFFu));
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (lane == 0) {
            const int e = row_scale_exponent(mx);
            s_e[c] = e;
            if (blockIdx.x == 0 && s_tok[c] >= 0) a.xe[s_tok[c]] = e;   // for the down kernel
        }
    }

    using Code = typename std::conditional<BITS == 8, uint4, uint2>::type;   // 16 codes
    constexpr int kRowBytes = BITS == 8 ? 1 : 2;                              // inputs per byte
    const ExpertView vg = is_shared ? expert_view(a.s_gate, 0, I, H, BITS) : expert_view(a.gate, it.expert, I, H, BITS);
    const ExpertView vu = is_shared ? expert_view(a.s_up, 0, I, H, BITS) : expert_view(a.up, it.expert, I, H, BITS);
    const size_t rstride = (size_t)H / kRowBytes;
    const int r0 = blockIdx.x * 16 + g, r1 = r0 + 8;
    const int gbeg = (warp * G) / 8, gend = ((warp + 1) * G) / 8;

    float acc_g[NT][4], acc_u[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc_g[j][q] = acc_u[j][q] = 0.f;

    constexpr int GB = 4;   // groups whose loads are issued together
    for (int gb = gbeg; gb < gend; gb += GB) {
        Code cg0[GB], cg1[GB], cu0[GB], cu1[GB];
        uint16_t sg[GB][2], bg[GB][2], su[GB][2], bu[GB][2];
#pragma unroll
        for (int i = 0; i < GB; ++i) {
            const int grp = gb + i;
            if (grp < gend) {
                const size_t co = ((size_t)grp * 64 + 16 * t) / kRowBytes;
                cg0[i] = __ldg(reinterpret_cast<const Code *>(vg.codes + (size_t)r0 * rstride + co));
                cg1[i] = __ldg(reinterpret_cast<const Code *>(vg.codes + (size_t)r1 * rstride + co));
                cu0[i] = __ldg(reinterpret_cast<const Code *>(vu.codes + (size_t)r0 * rstride + co));
                cu1[i] = __ldg(reinterpret_cast<const Code *>(vu.codes + (size_t)r1 * rstride + co));
                sg[i][0] = __ldg(vg.scales + (size_t)r0 * G + grp);
                sg[i][1] = __ldg(vg.scales + (size_t)r1 * G + grp);
                bg[i][0] = __ldg(vg.biases + (size_t)r0 * G + grp);
                bg[i][1] = __ldg(vg.biases + (size_t)r1 * G + grp);
                su[i][0] = __ldg(vu.scales + (size_t)r0 * G + grp);
                su[i][1] = __ldg(vu.scales + (size_t)r1 * G + grp);
                bu[i][0] = __ldg(vu.biases + (size_t)r0 * G + grp);
                bu[i][1] = __ldg(vu.biases + (size_t)r1 * G + grp);
            }
        }
#pragma unroll
        for (int i = 0; i < GB; ++i) {
            const int grp = gb + i;
            if (grp >= gend) break;
            const float s_g0 = bf16_bits_to_float(sg[i][0]), s_g1 = bf16_bits_to_float(sg[i][1]);
            const float s_u0 = bf16_bits_to_float(su[i][0]), s_u1 = bf16_bits_to_float(su[i][1]);
            constexpr float off = BITS == 8 ? -2176.f : -128.f;                  // b - 128 s (b - 2176 s)
            const float c_g0 = fmaf(off, s_g0, bf16_bits_to_float(bg[i][0]));
            const float c_g1 = fmaf(off, s_g1, bf16_bits_to_float(bg[i][1]));
            const float c_u0 = fmaf(off, s_u0, bf16_bits_to_float(bu[i][0]));
            const float c_u1 = fmaf(off, s_u1, bf16_bits_to_float(bu[i][1]));
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const uint4 *xr = s_x + (j * 8 + g) * rowu4 + grp * 8 + 2 * t;
                uint32_t bp[8];
                permute_b(xr[0], xr[1], bp);
                float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f}, dx[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (BITS == 8) {
                    group_mma_bf16_b8(cg0[i], cg1[i], bp, dg, dx, true);
                    group_mma_bf16_b8(cu0[i], cu1[i], bp, du, dx, false);
                } else {
                    group_mma<false>(cg0[i], cg1[i], bp, dg, dx, true);
                    group_mma<false>(cu0[i], cu1[i], bp, du, dx, false);
                }
                // rows: d[0], d[1] -> row g; d[2], d[3] -> row g+8
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
        const int c0 = j * 8 + 2 * t;
        s_red[warp][0][g][c0] = acc_g[j][0];
        s_red[warp][0][g][c0 + 1] = acc_g[j][1];
        s_red[warp][0][g + 8][c0] = acc_g[j][2];
        s_red[warp][0][g + 8][c0 + 1] = acc_g[j][3];
        s_red[warp][1][g][c0] = acc_u[j][0];
        s_red[warp][1][g][c0 + 1] = acc_u[j][1];
        s_red[warp][1][g + 8][c0] = acc_u[j][2];
        s_red[warp][1][g + 8][c0 + 1] = acc_u[j][3];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < 16 * NT * 8; idx += blockDim.x) {
        const int c = idx >> 4, row = idx & 15;
        const int f = c < kDecodeMaxTok ? s_slot[c] : -1;
        if (f < 0) continue;
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            gs += s_red[w][0][row][c];
            us += s_red[w][1][row][c];
        }
        const float hv = gs / (1.f + __expf(-gs)) * us, dn = pow2f(-s_e[c]);
        a.h[(size_t)f * I + blockIdx.x * 16 + row] = __half_as_ushort(__float2half_rn(hv * dn * dn));
    }
}

// ------------------------------------------------------------ down projection
//
// grid (H/64, max items); 128 threads, warp w owns rows [64 bx + 16 w, +16) of
// the down matrix over all of the intermediate dimension; writes the raw
// expert output y_e for each of the item's slots.
template <int NT, int BITS>
__global__ void __launch_bounds__(128) decode_down_kernel(ExpertArgs a)
{
    extern __shared__ uint4 s_h[];                 // [NT*8][I/8 + 1]
    __shared__ int s_tok[kDecodeMaxTok], s_slot[kDecodeMaxTok];
    if ((int)blockIdx.y >= __ldg(a.nwork + 0)) return;
    const WorkItem it = a.work[blockIdx.y];
    const int H = a.H, I = a.I, GI = I / kGroup, rowu4 = I / 8 + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const bool is_shared = it.expert == a.E;

    item_columns(a, it, s_tok, s_slot);
    __syncthreads();
    for (int idx = threadIdx.x; idx < NT * 8 * (I / 8); idx += blockDim.x) {
        const int c = idx / (I / 8), col = idx - c * (I / 8);
        const int f = c < kDecodeMaxTok ? s_slot[c] : -1;
        s_h[c * rowu4 + col] = f >= 0 ? *(reinterpret_cast<const uint4 *>(a.h + (size_t)f * I) + col)
                                      : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();

    using Code = typename std::conditional<BITS == 8, uint4, uint2>::type;   // 16 codes
    constexpr int kRowBytes = BITS == 8 ? 1 : 2;                              // inputs per byte
    const ExpertView vd = is_shared ? expert_view(a.s_down, 0, H, I, BITS) : expert_view(a.down, it.expert, H, I, BITS);
    const size_t rstride = (size_t)I / kRowBytes;
    const int rbase = blockIdx.x * 64 + warp * 16;
    const int r0 = rbase + g, r1 = r0 + 8;
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;

    constexpr int GB = 8;
    for (int gb = 0; gb < GI; gb += GB) {
        Code c0[GB], c1[GB];
        uint16_t sv[GB][2], bv[GB][2];
#pragma unroll
        for (int i = 0; i < GB; ++i) {
            const int grp = gb + i;
            if (grp < GI) {
                const size_t co = ((size_t)grp * 64 + 16 * t) / kRowBytes;
                c0[i] = __ldg(reinterpret_cast<const Code *>(vd.codes + (size_t)r0 * rstride + co));
                c1[i] = __ldg(reinterpret_cast<const Code *>(vd.codes + (size_t)r1 * rstride + co));
                sv[i][0] = __ldg(vd.scales + (size_t)r0 * GI + grp);
                sv[i][1] = __ldg(vd.scales + (size_t)r1 * GI + grp);
                bv[i][0] = __ldg(vd.biases + (size_t)r0 * GI + grp);
                bv[i][1] = __ldg(vd.biases + (size_t)r1 * GI + grp);
            }
        }
#pragma unroll
        for (int i = 0; i < GB; ++i) {
            const int grp = gb + i;
            if (grp >= GI) break;
            const float s0 = bf16_bits_to_float(sv[i][0]), s1 = bf16_bits_to_float(sv[i][1]);
            const float k0 = fmaf(-1024.f, s0, bf16_bits_to_float(bv[i][0]));   // b - 1024 s
            const float k1 = fmaf(-1024.f, s1, bf16_bits_to_float(bv[i][1]));
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const uint4 *hr = s_h + (j * 8 + g) * rowu4 + grp * 8 + 2 * t;
                uint32_t bp[8];
                permute_b(hr[0], hr[1], bp);
                float d[4] = {0.f, 0.f, 0.f, 0.f}, dx[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (BITS == 8) group_mma(c0[i], c1[i], bp, d, dx, true);
                else group_mma<true>(c0[i], c1[i], bp, d, dx, true);
                acc[j][0] = fmaf(s0, d[0], fmaf(k0, dx[0], acc[j][0]));
                acc[j][1] = fmaf(s0, d[1], fmaf(k0, dx[1], acc[j][1]));
                acc[j][2] = fmaf(s1, d[2], fmaf(k1, dx[2], acc[j][2]));
                acc[j][3] = fmaf(s1, d[3], fmaf(k1, dx[3], acc[j][3]));
            }
        }
    }
    // h was stored as h 2^-2e: the slot's output is scaled back by 2^2e (exact)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int cA = j * 8 + 2 * t, cB = cA + 1;
        const int fA = cA < kDecodeMaxTok ? s_slot[cA] : -1, fB = cB < kDecodeMaxTok ? s_slot[cB] : -1;
        if (fA >= 0) {
            const float up = pow2f(__ldg(a.xe + s_tok[cA]));
            a.yslot[(size_t)fA * H + r0] = acc[j][0] * up * up;
            a.yslot[(size_t)fA * H + r1] = acc[j][2] * up * up;
        }
        if (fB >= 0) {
            const float up = pow2f(__ldg(a.xe + s_tok[cB]));
            a.yslot[(size_t)fB * H + r0] = acc[j][1] * up * up;
            a.yslot[(size_t)fB * H + r1] = acc[j][3] * up * up;
        }
    }
}

// ------------------------------------------------------------ fixed-order slot sum
//
// sum[t, n] = sum_{j < k} p[t,j] * y_slot[t*k + j, n] + w_s[t] * y_slot[T*k + t, n],
// added in slot order; y = bf16(sum) or acc += sum.  One thread per 4 consecutive n of a token.
// Routed slot f sits in row pos[f] of the slot buffer (row f without pos).
__global__ void slot_sum_kernel(ReduceArgs a)
{
    const int H4 = a.H / 4, k = a.k, Tk = a.T * a.k;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)a.T * H4) return;
    const int t = (int)(idx / H4), n4 = (int)(idx - (size_t)t * H4);
    const float4 *ys = reinterpret_cast<const float4 *>(a.yslot);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float w, float4 v) {
        s.x = fmaf(w, v.x, s.x);
        s.y = fmaf(w, v.y, s.y);
        s.z = fmaf(w, v.z, s.z);
        s.w = fmaf(w, v.w, s.w);
    };
#pragma unroll 4
    for (int j = 0; j < k; ++j) {
        const int f = t * k + j;
        const int r = a.pos ? __ldg(a.pos + f) : f;
        if (r < 0 || r >= Tk) {                        // an inconsistent permutation: report, skip the slot
            record_status(a.status, MOE_ERR_DEVICE);
            continue;
        }
        add(bf16_bits_to_float(a.p[f]), __ldcs(ys + (size_t)r * H4 + n4));
    }
    if (a.has_shared) add(bf16_bits_to_float(a.w_s[t]), __ldcs(ys + ((size_t)Tk + t) * H4 + n4));
    if (a.y) {
        uint2 o;
        o.x = (uint32_t)float_to_bf16_bits(s.x) | ((uint32_t)float_to_bf16_bits(s.y) << 16);
        o.y = (uint32_t)float_to_bf16_bits(s.z) | ((uint32_t)float_to_bf16_bits(s.w) << 16);
        reinterpret_cast<uint2 *>(a.y)[idx] = o;
    } else {
        float4 *acc = reinterpret_cast<float4 *>(a.acc) + idx;
        float4 v = *acc;
        v.x += s.x;
        v.y += s.y;
        v.z += s.z;
        v.w += s.w;
        *acc = v;
    }
}

__global__ void invert_perm_kernel(const int32_t *__restrict__ perm, int32_t *__restrict__ inv, int n, int *status)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int f = perm[i];
    if (f < 0 || f >= n) record_status(status, MOE_ERR_DEVICE);
    else inv[f] = i;
}

// One thread per 4 consecutive columns of one output slot.
__global__ void slot_gather_kernel(const float4 *__restrict__ ys, const int32_t *__restrict__ pos, float4 *__restrict__ out,
                                   int T, int H4, int k, int has_shared, int *status)
{
    const int Tk = T * k, nslot = Tk + (has_shared ? T : 0);
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)nslot * H4) return;
    const int f = (int)(idx / H4), n4 = (int)(idx - (size_t)f * H4);
    const int r = f < Tk ? __ldg(pos + f) : f;
    if (r < 0 || r >= nslot) {
        record_status(status, MOE_ERR_DEVICE);
        return;
    }
    out[idx] = ys[(size_t)r * H4 + n4];
}

}  // namespace

namespace {

template <int NT, int BITS>
cudaError_t launch_gateup_as(const ExpertArgs &a, size_t smem, cudaStream_t st)
{
    cudaFuncSetAttribute(decode_gateup_kernel<NT, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    decode_gateup_kernel<NT, BITS><<<dim3(a.I / 16, a.max_items), 256, smem, st>>>(a);
    return cudaGetLastError();
}

template <int NT, int BITS>
cudaError_t launch_down_as(const ExpertArgs &a, size_t smem, cudaStream_t st)
{
    cudaFuncSetAttribute(decode_down_kernel<NT, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    decode_down_kernel<NT, BITS><<<dim3(a.H / 64, a.max_items), 128, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_gateup(const ExpertArgs &a, cudaStream_t st)
{
    const int ncol = a.T >= 9 ? 16 : 8;
    const size_t smem = (size_t)ncol * (a.H / 8 + 1) * 16;
    if (a.bits == 8) return ncol == 16 ? launch_gateup_as<2, 8>(a, smem, st) : launch_gateup_as<1, 8>(a, smem, st);
    return ncol == 16 ? launch_gateup_as<2, 4>(a, smem, st) : launch_gateup_as<1, 4>(a, smem, st);
}

cudaError_t launch_decode_down(const ExpertArgs &a, cudaStream_t st)
{
    const int ncol = a.T >= 9 ? 16 : 8;
    const size_t smem = (size_t)ncol * (a.I / 8 + 1) * 16;
    if (a.bits == 8) return ncol == 16 ? launch_down_as<2, 8>(a, smem, st) : launch_down_as<1, 8>(a, smem, st);
    return ncol == 16 ? launch_down_as<2, 4>(a, smem, st) : launch_down_as<1, 4>(a, smem, st);
}

cudaError_t launch_slot_sum(const ReduceArgs &a, cudaStream_t st)
{
    const size_t n = (size_t)a.T * (a.H / 4);
    slot_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_invert_perm(const int32_t *perm, int32_t *inv, int n, int *status, cudaStream_t st)
{
    if (n <= 0) return cudaSuccess;
    invert_perm_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(perm, inv, n, status);
    return cudaGetLastError();
}

cudaError_t launch_slot_gather(const float *yslot, const int32_t *pos, float *out, int T, int H, int k, int has_shared,
                               int *status, cudaStream_t st)
{
    const size_t n = (size_t)(T * k + (has_shared ? T : 0)) * (H / 4);
    if (n == 0) return cudaSuccess;
    slot_gather_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(reinterpret_cast<const float4 *>(yslot), pos,
                                                                     reinterpret_cast<float4 *>(out), T, H / 4, k,
                                                                     has_shared, status);
    return cudaGetLastError();
}

}  // namespace qmoe
