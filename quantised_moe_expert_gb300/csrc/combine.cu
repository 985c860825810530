// The single rounding of moe_combine: y = bf16_rne(acc).
#include "kernels.cuh"

namespace qmoe {
namespace {

__global__ void combine_kernel(const float4 *__restrict__ acc, uint2 *__restrict__ y, size_t n4)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = acc[i];
        uint2 o;
        o.x = (uint32_t)float_to_bf16_bits(v.x) | ((uint32_t)float_to_bf16_bits(v.y) << 16);
        o.y = (uint32_t)float_to_bf16_bits(v.z) | ((uint32_t)float_to_bf16_bits(v.w) << 16);
        y[i] = o;
    }
}

unsigned grid_for(size_t n)
{
    const size_t want = (n + 255) / 256;
    return (unsigned)(want < 152 * 16 ? (want ? want : 1) : 152 * 16);
}

}  // namespace

// n is a multiple of 4 (H is a multiple of 64).
cudaError_t launch_combine(const float *acc, uint16_t *y, size_t n, cudaStream_t st)
{
    combine_kernel<<<grid_for(n / 4), 256, 0, st>>>(reinterpret_cast<const float4 *>(acc),
                                                       reinterpret_cast<uint2 *>(y), n / 4);
    return cudaGetLastError();
}

}  // namespace qmoe
