// Shared device/host definitions of the MoE layer kernels (sm_103a).
#pragma once

#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace qmoe {

constexpr int kGroup = 64;          // quantisation group along the input dimension
constexpr int kMaxExperts = 256;    // top-k kernel keeps E/32 logits per lane
constexpr int kMaxTopK = 16;
constexpr int kMaxTokens = 65536;
constexpr int kTokBlock = 128;      // tokens per block of the histogram / stable scatter
constexpr int kDecodeMaxTok = 16;   // decode GEMV handles up to 16 tokens per expert per pass

// Tile of the prefill grouped GEMMs: 128 weight rows x up to kTileN tokens.
constexpr int kTileM = 128;
constexpr int kTileN1 = 128;        // tokens per tile, gate/up GEMM (two accumulators)
constexpr int kTileN2 = 256;        // tokens per tile, down GEMM
constexpr int kSmallN = 32;         // tokens per item of the small-tile GEMMs (experts of at most kSmallN tokens)
constexpr int kBigTok = kSmallN + 1;   // experts with at least this many tokens go to the tensor-memory GEMMs

// Workspace header (int offsets from the start of the workspace): the device status word, then
// the fused decode kernel's grid-wide counters, 128 bytes apart, and the epoch of its last
// launch.  The counters must be zero before a workspace's first use; the fused decode kernel
// leaves them zero when it ends and advances the epoch (the tag of the logits it publishes).
constexpr int kSyncUnits = 64;      // CTAs whose expert units are done
constexpr int kSyncExit = 96;       // CTAs that have left
constexpr int kSyncEpoch = 120;     // launches so far (wraps)
constexpr size_t kHeaderBytes = 512;
constexpr int kTraceStamps = 14;    // %globaltimer stamps per CTA of the fused decode kernel
constexpr int kTraceMaxCtas = 256;
constexpr int kDecodeSlice = 32;    // rows of the intermediate dimension per fused decode unit

// 4-bit codes for mma.sync: the 8 nibbles of a code word -> four fp16 pairs of the signed codes q - 8
// (exact), elements (0,4), (1,5), (2,6), (3,7) of the word.  A nibble at bits 0-3 or 4-7 of a 16-bit
// half lies inside the fp16 mantissa once the half is ORed with 1024 (0x6400): 1024 + q, or
// 1024 + 16 q, which one exact f16x2 add or fma maps to q - 8.  So a word costs four masks and a
// single shift (for the nibbles at bits 8-15); in the weight-streaming GEMMs the integer pipe, not the
// tensor pipe, is the bound.  The six constants (DequantK) reach the kernels as launch parameters: as
// literals the compiler rebuilds them in registers inside the loops, which costs the integer pipe
// about a third more.
struct DequantK {
    uint32_t lo, hi, one024, sub, mul, add;   // 0x000F000F, 0x00F000F0, 1024, 1032, 1/16, -72 (f16x2)
};
constexpr DequantK kDequantK{0x000F000Fu, 0x00F000F0u, 0x64006400u, 0x64086408u, 0x2C002C00u, 0xD480D480u};
__device__ __forceinline__ void nib8_signed(uint32_t u, uint32_t *r, const DequantK &k)
{
    const uint32_t v = u >> 8;
    r[0] = (u & k.lo) | k.one024;
    r[1] = (u & k.hi) | k.one024;
    r[2] = (v & k.lo) | k.one024;
    r[3] = (v & k.hi) | k.one024;
    // (1024 + q) - 1032 and (1024 + 16 q) / 16 - 72
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(r[0]) : "r"(k.sub));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(r[1]) : "r"(k.mul), "r"(k.add));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(r[2]) : "r"(k.sub));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(r[3]) : "r"(k.mul), "r"(k.add));
}

// One unit of work of a grouped kernel: an expert (E = shared) and a token range
// [tok0, tok0 + ntok) of its permuted slot list.
struct WorkItem {
    int expert;
    int tok0;
    int ntok;
    int pad;
};

// Offsets (bytes) of every scratch array inside the caller's workspace.
struct WsLayout {
    size_t status;     // header: int32 status word + fused decode counters (kHeaderBytes)
    size_t logits;     // f32 [T, E] (prefill) or u64 [T, E] (fused decode)
    size_t ids;        // i32 [T, k]
    size_t p;          // u16 [T, k]
    size_t w_s;        // u16 [T]
    size_t gamma;      // f32 [T] shared gate logit
    size_t hist;       // i32 [nblk, E]
    size_t counts;     // i32 [E]
    size_t offsets;    // i32 [E + 1]
    size_t perm;       // i32 [T*k]
    size_t inv_perm;   // i32 [T*k]
    size_t nwork;      // i32 [8]: decode items, gemm1 items, gemm2 items, big gemm1 / gemm2 items
    size_t trace;      // u64 [kTraceMaxCtas, kTraceStamps] fused decode timeline
    size_t work_dec;   // WorkItem [E + 1]
    size_t work_g1;    // WorkItem [max tiles gemm1]
    size_t work_g2;    // WorkItem [max tiles gemm2]
    size_t x16;        // fp16 [T, H] (prefill B operand)
    size_t xsum;       // f32 [T, H / 64] group sums of x16 (small-tile gate/up GEMM)
    size_t xe;         // i32 [T] prefill pre-scale exponents: x16 holds x' = x 2^-xe
    size_t hsum;       // f32 [T*k + T, I / 64] group sums of h (small-tile GEMMs)
    size_t h;          // fp16 [T*k + T, I] (decode: slot order; prefill: expert-sorted, K-permuted)
    size_t yslot;      // f32 [T*k + T, H] (decode kernels of shapes the fused kernel does not take)
    size_t dpart;      // f32 [T*k + T, I / 32, H] fused decode: raw down sums per column and slice
    size_t dhsum;      // f32 [T*k + T, I / 32] fused decode: sums of h per column and slice
    size_t acc;        // f32 [T, H] (prefill accumulation)
    size_t total;
    int nblk;
    int max_wd;
    int max_w1;
    int max_w2;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline int max_tiles(int T, int k, int E, int has_shared, int tile_n)
{
    // sum over active experts of ceil(c_e / n) <= (T*k) / n + (number of active experts),
    // and at most min(E, T*k) experts are active; plus the shared expert's ceil(T / n).
    const long long active = (long long)T * k < E ? (long long)T * k : E;
    long long t = (long long)T * k / tile_n + active + (has_shared ? (T + tile_n - 1) / tile_n : 0) + 1;
    return (int)t;
}

// Number of SMs of the current device, cached per device (atomics: calls may come from any host thread;
// devices beyond the cache are queried every time).
inline int device_sm_count()
{
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const bool cached = dev >= 0 && dev < kMaxDev;
    if (cached) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
    if (cached) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

inline WsLayout ws_layout(const moe_config &c, int T)
{
    WsLayout L{};
    const size_t H = c.hidden, I = c.inter, E = c.n_experts, k = c.top_k;
    const size_t Tz = T > 0 ? T : 1;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
    L.nblk = (int)((Tz + kTokBlock - 1) / kTokBlock);
    L.max_w1 = max_tiles((int)Tz, (int)k, (int)E, c.has_shared, kSmallN);   // bounds both item sizes
    L.max_w2 = L.max_w1;
    L.status = take(kHeaderBytes);
    L.logits = take(8 * Tz * E);     // fp32 logits, or the fused decode kernel's (logit, epoch) pairs
    L.ids = take(4 * Tz * k);
    L.p = take(2 * Tz * k);
    L.w_s = take(2 * Tz);
    L.gamma = take(4 * Tz);
    L.hist = take(4 * (size_t)L.nblk * E);
    L.counts = take(4 * E);
    L.offsets = take(4 * (E + 1));
    L.perm = take(4 * Tz * k);
    L.inv_perm = take(4 * Tz * k);
    L.nwork = take(32);
    L.trace = take(8 * (size_t)kTraceMaxCtas * kTraceStamps);
    L.max_wd = max_tiles((int)Tz, (int)k, (int)E, c.has_shared, kDecodeMaxTok);
    L.work_dec = take(sizeof(WorkItem) * (size_t)L.max_wd);
    L.work_g1 = take(sizeof(WorkItem) * (size_t)L.max_w1);
    L.work_g2 = take(sizeof(WorkItem) * (size_t)L.max_w2);
    L.x16 = take(2 * Tz * H);
    L.xsum = take(4 * Tz * (H / 64));
    L.xe = take(4 * Tz);
    L.hsum = take(4 * Tz * (k + 1) * (I / 64));
    L.h = take(2 * Tz * (k + 1) * I);
    L.yslot = take(4 * Tz * (k + 1) * H);
    L.acc = take(4 * Tz * H);
    const size_t Td = Tz <= (size_t)kDecodeMaxTok ? Tz : 0;   // the fused decode kernel takes T <= 16
    L.dpart = take(4 * Td * (k + 1) * (I / kDecodeSlice) * H);
    L.dhsum = take(4 * Td * (k + 1) * (I / kDecodeSlice));
    L.total = o;
    return L;
}

// Device-side status recording: first error wins, never traps.
__device__ __forceinline__ void record_status(int *status, int code)
{
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b)
{
    return __uint_as_float(((uint32_t)b) << 16);
}

// Round a float to bf16 bits, nearest-even (finite inputs).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Round a double to bf16 bits, nearest-even, with a single rounding (normal range).
// Drops the low 45 of the 52 fraction bits with round-half-even on the bit
// pattern, then the 7-bit-fraction double is exactly representable in fp32.
__device__ __forceinline__ uint16_t double_to_bf16_bits(double d)
{
    unsigned long long u = (unsigned long long)__double_as_longlong(d);
    unsigned long long lsb = (u >> 45) & 1ull;
    u += 0x0FFFFFFFFFFFull + lsb;     // 2^44 - 1 + lsb
    u &= ~((1ull << 45) - 1ull);
    float f = (float)__longlong_as_double((long long)u);
    return (uint16_t)(__float_as_uint(f) >> 16);
}

// 2^n as a float, exactly, for -149 <= n <= 127 (powers of two below 2^-126 are subnormal).
__device__ __forceinline__ float pow2f(int n)
{
    return n >= -126 ? __int_as_float((n + 127) << 23) : __int_as_float(1 << (n + 149));
}

// Exponent e of a token's pre-scale from the largest |x| of its row as bf16 magnitude bits (sign
// cleared): 2^e <= max |x| < 2^(e + 1), so x' = x 2^-e has max |x'| in [1, 2) (e = -126 for a row of
// zeros and subnormals).
__device__ __forceinline__ int row_scale_exponent(uint32_t max_bits)
{
    const int ef = (int)(max_bits >> 7);
    return ef == 0 ? -126 : ef - 127;
}

}  // namespace qmoe
