// Router GEMV of many tokens on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).
//
// The router is MLX affine 8-bit in groups of 64 (page "Qwen3.6-35B-A3B
// (qwen3_5_moe) on the native Metal engine: proposal and gate", slice "The
// family, plain decode": "the routers at 8 bits"), and the logits are fp32.
// At prefill sizes the router is a small GEMM, [E x H] x [H x T]; with CUDA
// cores it dominated the layer.  No weight is rounded here: an 8-bit code
// q = 16 q_hi + q_lo is split into two nibbles, each made an exact bf16
// integer (OR into the mantissa of 128.0, then subtract 128 exactly), and per
// group of 64 inputs
//   sum_j w_j x_j = s (16 sum q_hi x + sum q_lo x) + b sum x
// with sum x from an all-ones MMA chain; scale and bias apply in fp32.  (Keeping
// the 128 offset inside the MMA sums would cancel ~4 bits of the fp32
// accumulation afterwards; the logits must stay within ~1e-6 of the exact
// sum so the top-k agrees with an exact router away from near-ties.)
//
// K order: a 32-bit word holds inputs 0..3 of a chunk; the bit operations
// yield pairs (0,2) and (1,3), and the x fragment is permuted the same way.
#include "kernels.cuh"

namespace qmoe {
namespace {

constexpr int kRExp = 32;                  // experts per block
constexpr int kRTok = 32;                  // tokens per block (4 n8 tiles)

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16x2 (128 + n0, 128 + n1) -> (n0, n1), exact.
__device__ __forceinline__ uint32_t sub128(uint32_t v)
{
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&v);
    h = __hsub2(h, __floats2bfloat162_rn(128.f, 128.f));
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// grid (ceil(E/32), ceil(T/32)), 256 threads.  Warp w: experts e0 + 16 (w & 1) .. +15 over the groups of
// quarter w >> 1 of the input dimension, all 32 tokens; the four quarters' partial sums are added in a
// fixed order (quarter 0 first) through shared memory.  A token's logits never depend on the other tokens.
__global__ void __launch_bounds__(256) router_mma_kernel(RouterMmaArgs a)
{
    __shared__ float s_part[4][kRExp][kRTok + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int H = a.H, E = a.E, T = a.T, G = H / kGroup;
    const int et = warp & 1, kq = warp >> 1;
    const int ebase = blockIdx.x * kRExp + et * 16;
    const int tbase = blockIdx.y * kRTok;
    const int r0 = min(ebase + g, E - 1), r1 = min(ebase + g + 8, E - 1);   // clamped rows are not stored
    int tok[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) tok[j] = tbase + j * 8 + g;

    float acc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;

    const int gbeg = (kq * G) / 4, gend = ((kq + 1) * G) / 4;
    for (int grp = gbeg; grp < gend; ++grp) {
        // 16 codes (bytes 16t..16t+15 of the group) of rows g and g+8
        const uint4 c0 = __ldg(reinterpret_cast<const uint4 *>(a.codes + (size_t)r0 * H + grp * 64 + 16 * t));
        const uint4 c1 = __ldg(reinterpret_cast<const uint4 *>(a.codes + (size_t)r1 * H + grp * 64 + 16 * t));
        const float s0 = bf16_bits_to_float(__ldg(a.scales + (size_t)r0 * G + grp));
        const float s1 = bf16_bits_to_float(__ldg(a.scales + (size_t)r1 * G + grp));
        const float k0 = bf16_bits_to_float(__ldg(a.biases + (size_t)r0 * G + grp));
        const float k1 = bf16_bits_to_float(__ldg(a.biases + (size_t)r1 * G + grp));
        const uint32_t w0[4] = {c0.x, c0.y, c0.z, c0.w}, w1[4] = {c1.x, c1.y, c1.z, c1.w};
        // lo / hi nibble pairs: word m -> {(0,2), (1,3)} of inputs 16t + 4m .. +3
        uint32_t lo0[8], lo1[8], hi0[8], hi1[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            lo0[2 * m] = sub128((w0[m] & 0x000F000Fu) | 0x43004300u);
            lo0[2 * m + 1] = sub128(((w0[m] >> 8) & 0x000F000Fu) | 0x43004300u);
            hi0[2 * m] = sub128(((w0[m] >> 4) & 0x000F000Fu) | 0x43004300u);
            hi0[2 * m + 1] = sub128(((w0[m] >> 12) & 0x000F000Fu) | 0x43004300u);
            lo1[2 * m] = sub128((w1[m] & 0x000F000Fu) | 0x43004300u);
            lo1[2 * m + 1] = sub128(((w1[m] >> 8) & 0x000F000Fu) | 0x43004300u);
            hi1[2 * m] = sub128(((w1[m] >> 4) & 0x000F000Fu) | 0x43004300u);
            hi1[2 * m + 1] = sub128(((w1[m] >> 12) & 0x000F000Fu) | 0x43004300u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t b[8];
            if (tok[j] < T) {
                const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + (size_t)tok[j] * H + grp * 64 + 16 * t);
                const uint4 xa = __ldg(xp), xb = __ldg(xp + 1);
                const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    b[2 * m] = prmt(xw[2 * m], xw[2 * m + 1], 0x5410u);       // inputs (0, 2)
                    b[2 * m + 1] = prmt(xw[2 * m], xw[2 * m + 1], 0x7632u);   // inputs (1, 3)
                }
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) b[q] = 0;
            }
            float dl[4] = {0.f, 0.f, 0.f, 0.f}, dh[4] = {0.f, 0.f, 0.f, 0.f}, dx[4] = {0.f, 0.f, 0.f, 0.f};
            constexpr uint32_t ones = 0x3F803F80u;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                mma_bf16(dl, lo0[2 * m], lo1[2 * m], lo0[2 * m + 1], lo1[2 * m + 1], b[2 * m], b[2 * m + 1]);
                mma_bf16(dh, hi0[2 * m], hi1[2 * m], hi0[2 * m + 1], hi1[2 * m + 1], b[2 * m], b[2 * m + 1]);
                mma_bf16(dx, ones, ones, ones, ones, b[2 * m], b[2 * m + 1]);
            }
            // rows: d[0], d[1] -> expert g; d[2], d[3] -> expert g+8
            acc[j][0] = fmaf(s0, fmaf(16.f, dh[0], dl[0]), fmaf(k0, dx[0], acc[j][0]));
            acc[j][1] = fmaf(s0, fmaf(16.f, dh[1], dl[1]), fmaf(k0, dx[1], acc[j][1]));
            acc[j][2] = fmaf(s1, fmaf(16.f, dh[2], dl[2]), fmaf(k1, dx[2], acc[j][2]));
            acc[j][3] = fmaf(s1, fmaf(16.f, dh[3], dl[3]), fmaf(k1, dx[3], acc[j][3]));
        }
    }
    // partial sums of this quarter: [quarter][expert in block][token in block]
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int c = j * 8 + 2 * t;
        s_part[kq][et * 16 + g][c] = acc[j][0];
        s_part[kq][et * 16 + g][c + 1] = acc[j][1];
        s_part[kq][et * 16 + g + 8][c] = acc[j][2];
        s_part[kq][et * 16 + g + 8][c + 1] = acc[j][3];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kRExp * kRTok; i += blockDim.x) {
        const int el = i / kRTok, tl = i - el * kRTok;
        const int e = blockIdx.x * kRExp + el, tt = tbase + tl;
        if (e < E && tt < T) {
            float l = s_part[0][el][tl];
            l += s_part[1][el][tl];
            l += s_part[2][el][tl];
            l += s_part[3][el][tl];
            if (a.router_bias) l = l + __ldg(a.router_bias + e);   // one fp32 rounding
            a.logits[(size_t)tt * E + e] = l;
        }
    }
}

}  // namespace

cudaError_t launch_router_mma(const RouterMmaArgs &a, cudaStream_t st)
{
    dim3 grid((a.E + kRExp - 1) / kRExp, (a.T + kRTok - 1) / kRTok);
    router_mma_kernel<<<grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace qmoe
