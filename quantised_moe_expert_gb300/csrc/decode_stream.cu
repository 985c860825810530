// Streaming decode layer for T <= 16: one cooperative launch after the router GEMV.
//
// The decode cost is the bytes of the selected experts (page "POC for qwen3.5 /
// qwen3.6 support optimized for AGX Orin", Phase 1-4: the batch-1 "gemv MoE
// path"; "both stacks are now weight-BW bound").  At T = 1 those are ~16 MB,
// a few microseconds of HBM time, so the whole expert stage stays in one grid
// of co-resident CTAs (one per SM) and the data movement is the TMA engine's:
//   - the work is a list of units: gate/up units (expert, 16 rows of I, both
//     matrices, all of H) followed by down units (expert, 128 rows of H, all
//     of I); CTA c takes units c, c + grid, c + 2 grid, ...;
//   - a producer thread streams each unit's int4 codes with TMA (one 3D copy per
//     matrix: the 128-byte chunks of the unit's rows, 128-byte swizzled, so the
//     MMA fragment reads below hit no bank twice) and its scales and biases
//     with bulk copies into a ring of shared-memory slots, as far ahead as the
//     ring allows; down units are loaded before their inputs exist;
//   - the eight consumer warps, as one group (T <= 2) or as two groups of four
//     taking alternate units (T > 2), compute each unit from shared memory,
//     write its result to global memory, release the slot and publish the unit
//     in shared memory;
//   - a signal thread makes the published units visible GPU-wide (one fence
//     per batch) and counts them: gate/up units per expert, down units per
//     128-row block; the last down unit of a row block queues that block's
//     combine for this CTA's consumers.  Before that, in CTAs assigned a
//     token, its warp computes the token's pick weights and shared weight in
//     fp64 (a long dependent chain on this GPU); only the combine waits for
//     them.
// Phase 0 (every CTA): stage x (in the codes' k order) and its per-group sums
// in shared memory, redo the top-k from the fp32 logits (same comparisons as
// the top-k kernel), list the distinct experts (increasing id, shared expert
// last), their columns and the columns' tokens.
// Gate/up unit: split-K in a fixed partition (eight partials over the 128-byte
// code boxes, added in one order), h = silu(g) * u stored as fp16 in the codes'
// k order.  Down unit: one thread waits (bounded, with backoff) for the
// expert's gate/up units, the expert's h columns are staged in shared memory
// (in the place of x, which no unit needs any more) with their group sums, the
// raw expert output is written per slot.  Combine: y = bf16(sum_j p_j
// y_slot[t k + j] + w_s y_slot[T k + t]) in slot order, one rounding.
//
// Arithmetic (the GEMV of the decode path): over one group of 64 inputs
//     sum_j w_j x_j = s (sum_j (OFF + q_j) x_j) + (b - OFF s) sum_j x_j,
// OFF + q exact in the MMA operand type (bf16 128 + q for x, fp16 1024 + q for
// h), products on mma.sync m16n8k16 with fp32 accumulation, per-group scale and
// bias in fp32.  Every output element is one MMA column and every sum has one
// order: a token's result does not depend on the other tokens of the batch.
//
// Code size matters here as much as arithmetic: at T = 1 every SM runs each
// code path two or three times, so instruction fetch is part of the critical
// path.  The hot loops are unrolled over one 128-byte box (four groups) only,
// and the rarely run parts (routing, lists, producer, signals, combine) are
// separate functions.  Counters are zeroed by the kernel that precedes this
// launch.
#include <algorithm>

#include "kernels.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace qmoe {
namespace {

using namespace tc;

constexpr int kConsumerWarps = 8;
constexpr int kWarpProd = 8, kWarpSig = 9;
constexpr int kSThreads = 320;
constexpr int kCounterStride = 32;       // counters 128 bytes apart: pollers and writers do not share a line
constexpr int kMaxList = kMaxExperts + 1;
constexpr int kMaxSlots = 6;
constexpr int kRows1 = 16;               // rows of a gate/up unit
constexpr int kRows2 = 128;              // rows of a down unit
constexpr int kBox1 = kRows1 * 128;      // bytes of one 128-byte-wide code box of a gate/up unit
constexpr int kBox2 = kRows2 * 128;      // same, down unit
constexpr int kMaxRowBlocks = 64;        // H / 128 for H <= 8192
constexpr long long kDrainLimit = 1ll << 22;

struct StreamMaps {
    CUtensorMap g, u, d, sg, su, sd;     // int4 codes of gate, up, down (routed stacks, then the shared expert)
    // 1: 3D maps (128-byte chunk, row, chunk index), so that one copy brings every 128-byte box of a
    // unit's rows; 0: 2D maps, one copy per box
    int whole;
};

// Shared-memory geometry (bytes), fixed per (T, H, I) on the host.
struct StreamGeom {
    int R;                 // ring slots
    uint32_t slot;         // bytes per slot (multiple of 1024)
    int nb1;               // 128-byte boxes per gate/up code row (H / 256)
    uint32_t up_off, sc1_off, sb1, bytes1;
    int nb2;               // 128-byte boxes per down code row (I / 256)
    uint32_t sc2_off;
    uint32_t x_off, sumx_off, h_off, hs_off, red_off, dyn;
    int x_stride;          // uint4 per staged x row
    int h_stride;          // fp16 per staged h column
};

struct SSmem {
    int ids[kDecodeMaxTok][kMaxTopK];
    float lg[kDecodeMaxTok][kMaxTopK];     // fp32 logit of each pick
    float p[kDecodeMaxTok][kMaxTopK];
    float ws[kDecodeMaxTok];
    int cnt[kMaxList];                     // picks of each expert
    int lpos[kMaxList];                    // list position of each used expert
    int cfill[kMaxList];
    int list[kMaxList];
    int ncols[kMaxList];
    int colptr[kMaxList + 1];
    int colf[kDecodeMaxTok * (kMaxTopK + 1)];   // slot index f of each column, expert after expert
    int ctok[kDecodeMaxTok * (kMaxTopK + 1)];   // token of each column
    int nlist;
    int ready[2];                          // per consumer group
    int abort;
    int sig[2];                            // units finished by each consumer group (the signal thread reads them)
    int sig_done;                          // the signal thread has counted every unit
    int ncomb, ncomb_snap[2];              // combines queued for the consumers, and each group's snapshot
    int combq[kMaxRowBlocks];
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

// 8 nibbles -> four 16-bit pairs of (OFF + q), elements (0,4), (1,5), (2,6), (3,7).
template <bool F16>
__device__ __forceinline__ void nib8(uint32_t u, uint32_t *r)
{
    constexpr uint32_t base = F16 ? 0x64006400u : 0x43004300u;
    r[0] = (u & 0x000F000Fu) | base;
    r[1] = ((u >> 4) & 0x000F000Fu) | base;
    r[2] = ((u >> 8) & 0x000F000Fu) | base;
    r[3] = ((u >> 12) & 0x000F000Fu) | base;
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

// Position of input i in the k order of its chunk of 8.
__device__ __forceinline__ int kperm_pos(int i) { return (i & ~7) | ((i & 3) << 1) | ((i >> 2) & 1); }

// Byte offset, inside a row's 128-byte box, of the 8 code bytes that lane (g, t4) reads for group
// grp: 16-byte chunk 2 (grp % 4) + t4 / 2 of row r (r % 8 == g), stored at chunk index (chunk ^ g).
__device__ __forceinline__ uint32_t swz_chunk(int grp, int g, int t4)
{
    return (uint32_t)((((((grp & 3) << 1) | (t4 >> 1)) ^ g) << 4) | ((t4 & 1) << 3));
}

// Element q (0..3) of four bf16 values packed in a uint2, as a float.
__device__ __forceinline__ float bf16x4_at(uint2 v, int q)
{
    const uint32_t w = q < 2 ? v.x : v.y;
    return __uint_as_float((q & 1) ? (w & 0xFFFF0000u) : (w << 16));
}
__device__ __forceinline__ float f4_at(float4 v, int q) { return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w; }
__device__ __forceinline__ uint2 lds_u2(const uint16_t *p) { return *reinterpret_cast<const uint2 *>(p); }

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

// Bounded poll (backoff) until *cnt >= target; false when the limit ran out.
__device__ __forceinline__ bool poll_at_least(const int *cnt, int target, long long limit)
{
    long long n = 0;
    unsigned ns = 32;
    while (ld_acquire(cnt) < target) {
        if (++n > limit) return false;
        __nanosleep(ns);
        ns = ns < 512 ? ns * 2 : 512;
    }
    return true;
}

// Shared-memory flag accesses with CTA-scope acquire / release.
__device__ __forceinline__ int ld_acquire_cta(const int *p)
{
    int v;
    asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_cta(int *p, int v)
{
    asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// Named barriers of the consumer warps: 1 + g for consumer group g (CT threads), 3 for all
// consumer warps when there are two groups.
// (The ids are immediates, g being warp-uniform, so that a CTA reserves only the barriers it uses.)
template <int CT>
__device__ __forceinline__ void group_bar(int g)
{
    if (g == 0)
        asm volatile("bar.sync 1, %0;" ::"n"(CT) : "memory");
    else
        asm volatile("bar.sync 2, %0;" ::"n"(CT) : "memory");
}

// The group barrier that also ORs a predicate over the group (uniform stop decisions).
template <int CT>
__device__ __forceinline__ bool group_any(int g, bool pred)
{
    uint32_t r;
    if (g == 0)
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(r)
            : "r"((uint32_t)pred), "n"(CT)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 2, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(r)
            : "r"((uint32_t)pred), "n"(CT)
            : "memory");
    return r != 0;
}

__device__ __forceinline__ void all_consumers_bar() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

__device__ __forceinline__ int col_token(int f, int T, int k) { return f < 0 ? -1 : (f >= T * k ? f - T * k : f / k); }

// ------------------------------------------------------------------ phase 0 (all threads)
//
// x rows into shared memory in the codes' k order and their per-group sums (the caller's
// input only: this part overlaps the router kernel), then the routing (top-k of the fp32
// logits, or the caller's ids), the list of distinct experts and their columns.  The code
// is kept short: at T = 1 every SM fetches it cold, and that fetch is on the critical path.
__device__ __forceinline__ float key_logit(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__device__ __forceinline__ void phase0(SSmem &S, const FusedDecodeArgs &a, uint4 *s_x, float *s_sumx, int xs)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, H = a.H, E = a.E, k = a.k, G = H / kGroup, cpr = H / 8;
#pragma unroll 1
    for (int i = tid; i < T * cpr; i += kSThreads) {
        const int tt = i / cpr, col = i - tt * cpr;
        cp_async16(smem_u32(s_x + tt * xs + col), reinterpret_cast<const uint4 *>(a.x + (size_t)tt * H) + col);
    }
    cp_async_commit();
#pragma unroll 1
    for (int e = tid; e < kMaxList; e += kSThreads) {
        S.cnt[e] = 0;
        S.cfill[e] = 0;
    }
    cp_async_wait_all();
    __syncthreads();
#pragma unroll 1
    for (int i = tid; i < T * cpr; i += kSThreads) {
        const int tt = i / cpr, col = i - tt * cpr;
        s_x[tt * xs + col] = kperm8(s_x[tt * xs + col]);   // each chunk read and written by one thread
    }
    __syncthreads();
    // per-token sums of x over each group (fixed order; the bias term of the gate/up GEMV)
#pragma unroll 1
    for (int i = tid; i < T * G; i += kSThreads) {
        const int tt = i / G, grp = i - tt * G;
        const uint4 *xr = s_x + tt * xs + grp * 8;
        float sum = 0.f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
            const uint4 v = xr[c];
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                sum += __uint_as_float(w4[q] << 16);
                sum += __uint_as_float(w4[q] & 0xFFFF0000u);
            }
        }
        s_sumx[i] = sum;
    }

    // everything below reads what the preceding kernels wrote (logits, gamma, zeroed counters)
    pdl_wait();
    if (a.ids_in) {
#pragma unroll 1
        for (int i = tid; i < T * k; i += kSThreads) {
            const int tt = i / k, j = i - tt * k;
            int e = a.ids_in[i];
            if (e < 0 || e >= E) {
                record_status(a.status, MOE_ERR_DEVICE);
                e = 0;
            }
            S.ids[tt][j] = e;
            S.p[tt][j] = bf16_bits_to_float(a.p_in[i]);
            atomicAdd(&S.cnt[e], 1);
        }
#pragma unroll 1
        for (int tt = tid; tt < T; tt += kSThreads)
            S.ws[tt] = bf16_bits_to_float((a.has_shared && a.ws_in) ? a.ws_in[tt] : (uint16_t)0);
    } else {
        // one warp per token: lane l holds the keys of logits e = l + 32 r; each of the k rounds
        // takes the largest key (warp max), then the lowest id holding it (warp min), so the ids
        // come in rank order with equal logits going to the lower id
        constexpr int RW = kMaxExperts / 32;
#pragma unroll 1
        for (int tt = warp; tt < T; tt += kSThreads / 32) {
            uint32_t key[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int e = lane + 32 * r;
                key[r] = e < E ? logit_key(__ldg(a.logits + (size_t)tt * E + e)) : 0u;   // 0: below every logit
            }
#pragma unroll 1
            for (int j = 0; j < k; ++j) {
                uint32_t bk = key[0];
                int br = 0;
#pragma unroll
                for (int r = 1; r < RW; ++r)
                    if (key[r] > bk) {
                        bk = key[r];
                        br = r;
                    }
                const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
                const uint32_t mine = (uint32_t)(lane + 32 * br);
                const uint32_t id = __reduce_min_sync(0xffffffffu, bk == mk ? mine : 0xffffffffu);
                if (id == mine) {
#pragma unroll
                    for (int r = 0; r < RW; ++r)
                        if (r == br) key[r] = 0u;
                    S.ids[tt][j] = (int)id;
                    S.lg[tt][j] = key_logit(mk);
                    atomicAdd(&S.cnt[id], 1);
                }
            }
        }
    }
    __syncthreads();
    if (blockIdx.x == 0 && !a.ids_in && a.ids_out)
#pragma unroll 1
        for (int i = tid; i < T * k; i += kSThreads) a.ids_out[i] = S.ids[i / k][i % k];
    // the distinct experts in increasing id (list position lpos), their column counts and
    // offsets, then the shared expert's T columns
    if (warp == 0) {
        const int per = (E + 31) / 32, b0 = lane * per, b1 = min(E, b0 + per);
        int nloc = 0, cloc = 0;
#pragma unroll 1
        for (int e = b0; e < b1; ++e) {
            const int c = S.cnt[e];
            nloc += c > 0;
            cloc += c;
        }
        int ni = nloc, ci = cloc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vn = __shfl_up_sync(0xffffffffu, ni, o), vc = __shfl_up_sync(0xffffffffu, ci, o);
            if (lane >= o) {
                ni += vn;
                ci += vc;
            }
        }
        int pos = ni - nloc, col = ci - cloc;
#pragma unroll 1
        for (int e = b0; e < b1; ++e) {
            const int c = S.cnt[e];
            if (c > 0) {
                if (c > T) record_status(a.status, MOE_ERR_DEVICE);   // an id repeated within a token
                S.list[pos] = e;
                S.lpos[e] = pos;
                S.ncols[pos] = c;
                S.colptr[pos] = col;
                ++pos;
                col += c;
            }
        }
        if (lane == 31) {
            int D = ni;
            if (a.has_shared) {
                S.list[D] = E;
                S.ncols[D] = T;
                S.colptr[D] = ci;
                ++D;
            }
            S.colptr[D] = ci + (a.has_shared ? T : 0);
            S.nlist = D;
        }
    }
    __syncthreads();
    // columns of each expert: its slots (in no particular order: every column is computed on
    // its own), the shared expert's in token order
#pragma unroll 1
    for (int i = tid; i < T * k; i += kSThreads) {
        const int d = S.lpos[S.ids[i / k][i % k]];
        S.colf[S.colptr[d] + atomicAdd(&S.cfill[d], 1)] = i;
    }
    if (a.has_shared)
#pragma unroll 1
        for (int tt = tid; tt < T; tt += kSThreads) S.colf[S.colptr[S.nlist - 1] + tt] = T * k + tt;
    __syncthreads();
#pragma unroll 1
    for (int i = tid; i < S.colptr[S.nlist]; i += kSThreads) S.ctok[i] = col_token(S.colf[i], T, k);
    __syncthreads();
}

// ------------------------------------------------------------------ producer (one thread)
__device__ __noinline__ void producer(SSmem &S, const StreamMaps &maps, const FusedDecodeArgs &a,
                                      const StreamGeom &geo, uint8_t *ring, int U1, int U)
{
    // Every argument the loop needs, read once into registers: the arguments are reached through
    // references here, and each copy instruction below is a compiler memory barrier, so fields
    // read inside the loop would be fetched again after every copy.
    const int H = a.H, I = a.I, E = a.E, G = H / kGroup, GI = I / kGroup, R = geo.R;
    const int RBI = I / kRows1, RBH = (H + kRows2 - 1) / kRows2;
    const int nb1 = geo.nb1, nb2 = geo.nb2;
    const uint32_t slot_bytes = geo.slot, up_off = geo.up_off, sc1_off = geo.sc1_off, sb1 = geo.sb1;
    const uint32_t bytes1 = geo.bytes1, sc2_off = geo.sc2_off;
    const long long wait_limit = a.wait_limit;
    const uint16_t *gsc = a.gate.scales, *gbi = a.gate.biases, *usc = a.up.scales, *ubi = a.up.biases;
    const uint16_t *dsc = a.down.scales, *dbi = a.down.biases;
    const uint16_t *sgsc = a.s_gate.scales, *sgbi = a.s_gate.biases, *susc = a.s_up.scales, *subi = a.s_up.biases;
    const uint16_t *sdsc = a.s_down.scales, *sdbi = a.s_down.biases;
    const CUtensorMap *mg_r = &maps.g, *mu_r = &maps.u, *md_r = &maps.d;
    const CUtensorMap *mg_s = &maps.sg, *mu_s = &maps.su, *md_s = &maps.sd;
    const bool whole = maps.whole != 0;
    prefetch_map(mg_r);
    prefetch_map(mu_r);
    prefetch_map(md_r);
    if (a.has_shared) {
        prefetch_map(mg_s);
        prefetch_map(mu_s);
        prefetch_map(md_s);
    }
    int issued = 0;
#pragma unroll 1
    for (int w = blockIdx.x, i = 0; w < U; w += gridDim.x, ++i) {
        const int slot = i % R;
        if (i >= R && !mbar_wait_sleepy(smem_u32(&S.empty[slot]), ((i / R) - 1) & 1, wait_limit, &S.abort)) {
            S.abort = 1;
            record_status(a.status, MOE_ERR_TIMEOUT);
            break;
        }
        uint8_t *base = ring + (size_t)slot * slot_bytes;
        const uint32_t fb = smem_u32(&S.full[slot]);
        // this unit into the slot
        if (w < U1) {
            const int d = w / RBI, rb = w - d * RBI, e = S.list[d];
            const bool shr = e == E;
            const int row0 = (shr ? 0 : e * I) + rb * kRows1;
            const size_t so = (size_t)row0 * G;
            const CUtensorMap *mg = shr ? mg_s : mg_r, *mu = shr ? mu_s : mu_r;
            mbar_arrive_expect_tx(fb, bytes1);
            if (whole) {
                tma_load_3d(smem_u32(base), mg, 0, row0, 0, fb);
                tma_load_3d(smem_u32(base + up_off), mu, 0, row0, 0, fb);
            } else {
#pragma unroll 1
                for (int j = 0; j < nb1; ++j) {
                    tma_load_2d(smem_u32(base + j * kBox1), mg, j * 128, row0, fb);
                    tma_load_2d(smem_u32(base + up_off + j * kBox1), mu, j * 128, row0, fb);
                }
            }
            bulk_load(smem_u32(base + sc1_off), (shr ? sgsc : gsc) + so, sb1, fb);
            bulk_load(smem_u32(base + sc1_off + sb1), (shr ? sgbi : gbi) + so, sb1, fb);
            bulk_load(smem_u32(base + sc1_off + 2 * sb1), (shr ? susc : usc) + so, sb1, fb);
            bulk_load(smem_u32(base + sc1_off + 3 * sb1), (shr ? subi : ubi) + so, sb1, fb);
        } else {
            const int v = w - U1, d = v / RBH, rb = v - d * RBH, e = S.list[d];
            const bool shr = e == E;
            const int row0 = (shr ? 0 : e * H) + rb * kRows2;
            const int nrows = min(kRows2, H - rb * kRows2);
            const uint32_t sb2 = (uint32_t)nrows * GI * 2;
            const size_t so = (size_t)row0 * GI;
            const CUtensorMap *md = shr ? md_s : md_r;
            mbar_arrive_expect_tx(fb, (uint32_t)nb2 * kBox2 + 2 * sb2);
            if (whole) {
                tma_load_3d(smem_u32(base), md, 0, row0, 0, fb);
            } else {
#pragma unroll 1
                for (int j = 0; j < nb2; ++j) tma_load_2d(smem_u32(base + j * kBox2), md, j * 128, row0, fb);
            }
            bulk_load(smem_u32(base + sc2_off), (shr ? sdsc : dsc) + so, sb2, fb);
            bulk_load(smem_u32(base + sc2_off + kRows2 * GI * 2), (shr ? sdbi : dbi) + so, sb2, fb);
        }
        issued = i + 1;
    }
    // every issued copy lands before the CTA may exit
#pragma unroll 1
    for (int q = issued > R ? issued - R : 0; q < issued; ++q)
        mbar_wait(smem_u32(&S.full[q % R]), (q / R) & 1, kDrainLimit, nullptr);
}

// ------------------------------------------------------------------ signal warp
//
// First, in the CTA assigned token grid - 1 - blockIdx, the token's pick weights p =
// exp(l - l_top) / sum over the picks and w_s = sigmoid(bf16(gamma)) in fp64, one rounding
// to bf16, published for the combining CTAs.  Then (lane 0) the completion signals of
// this CTA's units.
template <int CG>
__device__ __noinline__ void signaller(SSmem &S, const FusedDecodeArgs &a, int U1, int U, int D)
{
    const int lane = threadIdx.x & 31, T = a.T, k = a.k, H = a.H, I = a.I;
    const int RBI = I / kRows1, RBH = (H + kRows2 - 1) / kRows2;
    const int tt = (int)gridDim.x - 1 - (int)blockIdx.x;
    if (!a.ids_in && tt >= 0 && tt < T) {
        double ex = 0.0;
        if (lane < k) ex = exp((double)S.lg[tt][lane] - (double)S.lg[tt][0]);
        double den = 0.0;
        #pragma unroll 1
        for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, ex, j);   // fixed order j = 0..k-1
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
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            atomicAdd(a.cnt_pick, 1);
        }
    }
    if (lane != 0) return;
    int *const cnt_expert = a.cnt_expert, *const cnt_rows = a.cnt_rows;   // read once (see the producer)
    const int *const cnt_pick = a.cnt_pick;
    const long long wait_limit = a.wait_limit;
    // Consumer group g takes this CTA's units g, g + CG, g + 2 CG, ... and publishes how many it
    // has finished in S.sig[g] (release at CTA scope).  One fence makes a batch of units' global
    // stores visible GPU-wide, then each unit is counted.
    const int nmine = (int)blockIdx.x < U ? (U - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    int done = 0, nq = 0, gdone0 = 0, gdone1 = 0;
    bool picks = a.ids_in != nullptr;       // given routing: S.p and S.ws were filled in phase 0
    // the published pick weights into shared memory (once every token's are out), for the combines
    auto take_picks = [&]() {
#pragma unroll 1
        for (int tt = 0; tt < T; ++tt)
#pragma unroll 1
            for (int j = 0; j < k; ++j) S.p[tt][j] = bf16_bits_to_float(__ldcg(a.p_glob + tt * k + j));
        #pragma unroll 1
        for (int q = 0; q < T; ++q) S.ws[q] = bf16_bits_to_float(__ldcg(a.ws_glob + q));
    };
    long long polls = 0;
    while (done < nmine) {
        const int avail0 = ld_acquire_cta(&S.sig[0]), avail1 = CG > 1 ? ld_acquire_cta(&S.sig[1]) : 0;
        const int fresh = (avail0 - gdone0) + (avail1 - gdone1);
        if (fresh <= 0) {
            if (S.abort || ++polls > wait_limit) break;
            if (!picks && ld_acquire(cnt_pick) >= T) {   // idle: fetch the pick weights ahead of any combine
                take_picks();
                picks = true;
            }
            __nanosleep(64);
            continue;
        }
        polls = 0;
        __threadfence();
        #pragma unroll 1
        for (int q = 0; q < fresh; ++q, ++done) {
            // the next finished unit: group 0's first, then group 1's
            const bool g0 = gdone0 < avail0;
            const int ui = g0 ? CG * gdone0++ : 1 + CG * gdone1++;
            const int w = (int)blockIdx.x + ui * (int)gridDim.x;
            if (w < U1) {
                atomicAdd(cnt_expert + (w / RBI) * kCounterStride, 1);
                continue;
            }
            const int rb = (w - U1) % RBH;
            if (atomicAdd(cnt_rows + rb * kCounterStride, 1) != D - 1) continue;
            __threadfence();                  // every unit's slot outputs, before the combine reads them
            if (!picks) {
                picks = poll_at_least(cnt_pick, T, wait_limit);
                if (picks) take_picks();
                else record_status(a.status, MOE_ERR_TIMEOUT);
            }
            if (picks && nq < kMaxRowBlocks) {
                S.combq[nq] = rb;
                st_release_cta(&S.ncomb, ++nq);
            }
        }
    }
    if (done < nmine) record_status(a.status, MOE_ERR_TIMEOUT);
    st_release_cta(&S.sig_done, 1);
}

// ------------------------------------------------------------------ combine (consumer warps)
//
// Row block rb of y (or acc): sum over the token's slots in slot order, one rounding.  The
// pick weights are in shared memory: the signal thread filled them before queueing the block.
template <int CT>
__device__ __noinline__ void combine_block(SSmem &S, const FusedDecodeArgs &a, int rb, int gid)
{
    const int gt = threadIdx.x - gid * CT, T = a.T, H = a.H, k = a.k;
    const bool has_shared = a.has_shared != 0;
    const float *const yslot = a.yslot;       // arguments read once (see the producer)
    uint16_t *const y = a.y;
    float *const acc = a.acc;
    const int nrow = min(kRows2, H - rb * kRows2), n4 = nrow / 4;   // H is a multiple of 64
    // four consecutive rows per thread: 16-byte loads, every load in flight before the first add
#pragma unroll 1
    for (int q = gt; q < n4 * T; q += CT) {
        const int tt = q / n4, row = rb * kRows2 + 4 * (q - tt * n4);
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 ysh = has_shared ? __ldcg(reinterpret_cast<const float4 *>(yslot + ((size_t)T * k + tt) * H + row)) : z;
        float4 sum = z;
        // the picks in order j = 0, 1, ..., eight slots' loads in flight at a time
#pragma unroll 1
        for (int jb = 0; jb < k; jb += 8) {
            float4 ys[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                ys[j] = jb + j < k ? __ldcg(reinterpret_cast<const float4 *>(yslot + ((size_t)tt * k + jb + j) * H + row)) : z;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (jb + j < k) {
                    const float pj = S.p[tt][jb + j];
                    sum.x = fmaf(pj, ys[j].x, sum.x);
                    sum.y = fmaf(pj, ys[j].y, sum.y);
                    sum.z = fmaf(pj, ys[j].z, sum.z);
                    sum.w = fmaf(pj, ys[j].w, sum.w);
                }
        }
        if (has_shared) {
            const float wsv = S.ws[tt];
            sum.x = fmaf(wsv, ysh.x, sum.x);
            sum.y = fmaf(wsv, ysh.y, sum.y);
            sum.z = fmaf(wsv, ysh.z, sum.z);
            sum.w = fmaf(wsv, ysh.w, sum.w);
        }
        if (y) {
            const uint32_t lo = (uint32_t)float_to_bf16_bits(sum.x) | ((uint32_t)float_to_bf16_bits(sum.y) << 16);
            const uint32_t hi = (uint32_t)float_to_bf16_bits(sum.z) | ((uint32_t)float_to_bf16_bits(sum.w) << 16);
            *reinterpret_cast<uint2 *>(y + (size_t)tt * H + row) = make_uint2(lo, hi);
        } else {
            float4 *ap = reinterpret_cast<float4 *>(acc + (size_t)tt * H + row);
            float4 av = *ap;
            av.x += sum.x;
            av.y += sum.y;
            av.z += sum.z;
            av.w += sum.w;
            *ap = av;
        }
    }
    group_bar<CT>(gid);
}

// ------------------------------------------------------------------ kernel
//
// CG consumer groups of 8 / CG warps: group g computes this CTA's units g, g + CG, ...
// With two groups one group's per-unit latencies (waits, barriers, the epilogue, the h
// exchange) overlap the other group's arithmetic.  The staged h columns of the down units
// share their shared memory with x: a group stages h only once both groups are past their
// last gate/up unit.
template <int NT, int MINB, int CG>
__global__ void __launch_bounds__(kSThreads, MINB)
    decode_stream_kernel(const __grid_constant__ StreamMaps maps, const __grid_constant__ FusedDecodeArgs a,
                         const __grid_constant__ StreamGeom geo)
{
    constexpr int CW = kConsumerWarps / CG, CT = CW * 32;   // warps and threads per consumer group
    constexpr int RT = kRows2 / (16 * CW);                  // 16-row tiles per warp in a down unit
    __shared__ SSmem S;
    extern __shared__ uint8_t dyn_raw[];
    uint8_t *dyn = align_smem_1024(dyn_raw);
    uint8_t *ring = dyn;
    uint4 *s_x = reinterpret_cast<uint4 *>(dyn + geo.x_off);          // [T][x_stride] bf16 rows, k order
    float *s_sumx = reinterpret_cast<float *>(dyn + geo.sumx_off);    // [T][G]
    float *s_red = reinterpret_cast<float *>(dyn + geo.red_off);      // [CG][8][2][16][NT * 8] split-K partials

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int T = a.T, H = a.H, I = a.I;
    const int G = H / kGroup, GI = I / kGroup, xs = geo.x_stride, R = geo.R;
    const long long limit = a.wait_limit;

    if (tid == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(smem_u32(&S.full[s]), 1);
            mbar_init(smem_u32(&S.empty[s]), CT);   // one group consumes each unit
        }
        S.abort = 0;
        S.sig[0] = S.sig[1] = 0;
        S.sig_done = 0;
        S.ncomb = 0;
        fence_mbar_init();
    }
    phase0(S, a, s_x, s_sumx, xs);

    const int D = S.nlist;
    const int RBI = I / kRows1, RBH = (H + kRows2 - 1) / kRows2;
    const int U1 = D * RBI, U = U1 + D * RBH;

    if (warp == kWarpProd) {
        if (lane == 0) producer(S, maps, a, geo, ring, U1, U);
        return;
    }
    if (warp == kWarpSig) {
        signaller<CG>(S, a, U1, U, D);
        return;
    }

    // ---------------------------------------------------------------- consumers (warps 0-7)
    constexpr int NC = NT * 8;
    const int gid = warp / CW, gw = warp - gid * CW, gt = tid - gid * CT;
    uint16_t *s_h = reinterpret_cast<uint16_t *>(dyn + geo.h_off) + (size_t)gid * NC * geo.h_stride;   // [NC][h_stride]
    float *s_hs = reinterpret_cast<float *>(dyn + geo.hs_off) + gid * NC * GI;                        // [NC][I / 64]
    int ncomb_done = gid;               // this group runs the queued combines gid, gid + CG, ...
    bool past_gateup = false;           // both groups are past their gate/up units (h may replace x)
    auto run_combines = [&](int snap) {
        for (; ncomb_done < snap; ncomb_done += CG) combine_block<CT>(S, a, S.combq[ncomb_done], gid);
    };

    for (int w = blockIdx.x + gid * (int)gridDim.x, i = gid; w < U; w += CG * (int)gridDim.x, i += CG) {
        const int slot = i % R;
        const bool got = mbar_wait(smem_u32(&S.full[slot]), (i / R) & 1, limit, &S.abort);
        if (!got) {
            S.abort = 1;
            record_status(a.status, MOE_ERR_TIMEOUT);
        }
        if (gt == 0) S.ncomb_snap[gid] = ld_acquire_cta(&S.ncomb);
        if (group_any<CT>(gid, !got)) break;
        run_combines(S.ncomb_snap[gid]);
        const uint8_t *base = ring + (size_t)slot * geo.slot;
        const uint32_t eb = smem_u32(&S.empty[slot]);

        if (w < U1) {
            // ------------------------------------------------ gate/up unit: 16 rows, split-K over the group's warps
            const int d = w / RBI, rb = w - d * RBI;
            const int ncol = min(S.ncols[d], T);
            const int *colf = S.colf + S.colptr[d], *ctok = S.ctok + S.colptr[d];
            int xrow[NT], tA[NT], tB[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int c = j * 8 + g, cA = j * 8 + 2 * t4;
                xrow[j] = c < ncol ? ctok[c] : -1;
                tA[j] = cA < ncol ? ctok[cA] : -1;
                tB[j] = cA + 1 < ncol ? ctok[cA + 1] : -1;
            }
            const uint16_t *gs = reinterpret_cast<const uint16_t *>(base + geo.sc1_off) + g * G;
            const uint16_t *gbi = gs + kRows1 * G, *us = gbi + kRows1 * G, *ubi = us + kRows1 * G;
            const uint8_t *cb = base + g * 128;          // row g of box 0; row g + 8 is 1024 bytes further
            // Split-K in a fixed partition whatever the number of groups: partial v (0..7) is the sum over
            // the 128-byte code boxes v, v + 8, ... (four groups of both matrices per box), and the
            // partials are added in the order v = 0..7.  Warp gw of the group computes the partials
            // gw, gw + CW, ...; a token's h is thus the same in every batch.
            float *red = s_red + (size_t)gid * kConsumerWarps * 2 * 16 * NC;   // [8][2][16][NC]
            float last[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
            for (int v = gw; v < kConsumerWarps; v += CW) {
                float acc_g[NT][4], acc_u[NT][4];
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc_g[j][q] = acc_u[j][q] = 0.f;
                // one box per step, unrolled so that every shared-memory load of a box is in flight before
                // its first MMA
#pragma unroll 1
                for (int bx = v; bx < geo.nb1; bx += kConsumerWarps) {
                    const uint2 vsg0 = lds_u2(gs + 4 * bx), vsg1 = lds_u2(gs + 8 * G + 4 * bx);
                    const uint2 vbg0 = lds_u2(gbi + 4 * bx), vbg1 = lds_u2(gbi + 8 * G + 4 * bx);
                    const uint2 vsu0 = lds_u2(us + 4 * bx), vsu1 = lds_u2(us + 8 * G + 4 * bx);
                    const uint2 vbu0 = lds_u2(ubi + 4 * bx), vbu1 = lds_u2(ubi + 8 * G + 4 * bx);
                    float4 sxA[NT], sxB[NT];                  // sums of x over the box's four groups
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                        sxA[j] = tA[j] >= 0 ? *reinterpret_cast<const float4 *>(s_sumx + tA[j] * G + 4 * bx) : z;
                        sxB[j] = tB[j] >= 0 ? *reinterpret_cast<const float4 *>(s_sumx + tB[j] * G + 4 * bx) : z;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int grp = 4 * bx + q;
                        const uint32_t o = (uint32_t)bx * kBox1 + swz_chunk(q, g, t4);
                        const uint2 cg0 = *reinterpret_cast<const uint2 *>(cb + o);
                        const uint2 cg1 = *reinterpret_cast<const uint2 *>(cb + o + 1024);
                        const uint2 cu0 = *reinterpret_cast<const uint2 *>(cb + geo.up_off + o);
                        const uint2 cu1 = *reinterpret_cast<const uint2 *>(cb + geo.up_off + o + 1024);
                        const float s_g0 = bf16x4_at(vsg0, q), s_g1 = bf16x4_at(vsg1, q);
                        const float s_u0 = bf16x4_at(vsu0, q), s_u1 = bf16x4_at(vsu1, q);
                        const float c_g0 = fmaf(-128.f, s_g0, bf16x4_at(vbg0, q));
                        const float c_g1 = fmaf(-128.f, s_g1, bf16x4_at(vbg1, q));
                        const float c_u0 = fmaf(-128.f, s_u0, bf16x4_at(vbu0, q));
                        const float c_u1 = fmaf(-128.f, s_u1, bf16x4_at(vbu1, q));
                        uint32_t ag[2][8], au[2][8];
                        nib8<false>(cg0.x, ag[0]);
                        nib8<false>(cg0.y, ag[0] + 4);
                        nib8<false>(cg1.x, ag[1]);
                        nib8<false>(cg1.y, ag[1] + 4);
                        nib8<false>(cu0.x, au[0]);
                        nib8<false>(cu0.y, au[0] + 4);
                        nib8<false>(cu1.x, au[1]);
                        nib8<false>(cu1.y, au[1] + 4);
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            if (j * 8 >= ncol) break;
                            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
                            if (xrow[j] >= 0) {
                                const uint4 *xr = s_x + xrow[j] * xs + grp * 8 + 2 * t4;
                                lo = xr[0];
                                hi = xr[1];
                            }
                            const uint32_t bp[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                            float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                mma16816<false>(dg, ag[0][2 * m], ag[1][2 * m], ag[0][2 * m + 1], ag[1][2 * m + 1], bp[2 * m],
                                                bp[2 * m + 1]);
                                mma16816<false>(du, au[0][2 * m], au[1][2 * m], au[0][2 * m + 1], au[1][2 * m + 1], bp[2 * m],
                                                bp[2 * m + 1]);
                            }
                            const float sA = f4_at(sxA[j], q), sB = f4_at(sxB[j], q);
                            acc_g[j][0] = fmaf(s_g0, dg[0], fmaf(c_g0, sA, acc_g[j][0]));
                            acc_g[j][1] = fmaf(s_g0, dg[1], fmaf(c_g0, sB, acc_g[j][1]));
                            acc_g[j][2] = fmaf(s_g1, dg[2], fmaf(c_g1, sA, acc_g[j][2]));
                            acc_g[j][3] = fmaf(s_g1, dg[3], fmaf(c_g1, sB, acc_g[j][3]));
                            acc_u[j][0] = fmaf(s_u0, du[0], fmaf(c_u0, sA, acc_u[j][0]));
                            acc_u[j][1] = fmaf(s_u0, du[1], fmaf(c_u0, sB, acc_u[j][1]));
                            acc_u[j][2] = fmaf(s_u1, du[2], fmaf(c_u1, sA, acc_u[j][2]));
                            acc_u[j][3] = fmaf(s_u1, du[3], fmaf(c_u1, sB, acc_u[j][3]));
                        }
                    }
                }
                float *rg = red + (v * 2 + 0) * 16 * NC, *ru = rg + 16 * NC;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int c0 = j * 8 + 2 * t4;
                    rg[g * NC + c0] = acc_g[j][0];
                    rg[g * NC + c0 + 1] = acc_g[j][1];
                    rg[(g + 8) * NC + c0] = acc_g[j][2];
                    rg[(g + 8) * NC + c0 + 1] = acc_g[j][3];
                    ru[g * NC + c0] = acc_u[j][0];
                    ru[g * NC + c0 + 1] = acc_u[j][1];
                    ru[(g + 8) * NC + c0] = acc_u[j][2];
                    ru[(g + 8) * NC + c0 + 1] = acc_u[j][3];
                }
                last[0] = acc_g[0][0];
                last[1] = acc_g[0][2];
                last[2] = acc_u[0][0];
                last[3] = acc_u[0][2];
            }
            mbar_arrive_after(eb, last[0], last[1], last[2], last[3]);
            group_bar<CT>(gid);
            // the partial sums in a fixed order, h = silu(g) u stored as fp16 in the
            // codes' k order (so the down unit's fragments are plain loads)
#pragma unroll 1
            for (int q = gt; q < 16 * ncol; q += CT) {
                const int row = q & 15, c = q >> 4;
                float gsum = 0.f, usum = 0.f;
#pragma unroll
                for (int v = 0; v < kConsumerWarps; ++v) {
                    gsum += red[((v * 2 + 0) * 16 + row) * NC + c];
                    usum += red[((v * 2 + 1) * 16 + row) * NC + c];
                }
                const float hv = gsum / (1.f + __expf(-gsum)) * usum;
                a.h[(size_t)colf[c] * I + kperm_pos(rb * kRows1 + row)] = __half_as_ushort(__float2half_rn(hv));
            }
            group_bar<CT>(gid);
            if (gt == 0) st_release_cta(&S.sig[gid], (i - gid) / CG + 1);
        } else {
            // ------------------------------------------------ down unit: 128 rows, RT 16-row tiles per warp
            if (CG > 1 && !past_gateup) {
                all_consumers_bar();          // x is dead from here on: h takes its place
                past_gateup = true;
            }
            const int v = w - U1, d = v / RBH, rb = v - d * RBH;
            const int ncol = min(S.ncols[d], T);
            const int *colf = S.colf + S.colptr[d];
            if (gt == 0) {
                const bool ok = poll_at_least(a.cnt_expert + d * kCounterStride, RBI, limit);
                if (!ok) {
                    S.abort = 1;
                    record_status(a.status, MOE_ERR_TIMEOUT);
                }
                S.ready[gid] = ok;
            }
            group_bar<CT>(gid);
            if (!S.ready[gid]) {
                mbar_arrive(eb);
                break;
            }
            // the expert's h columns into shared memory (L2 reads, after the acquire above), and each
            // column's sums over the groups of those fp16 values: 8 values per thread, then a shuffle
            // tree over the group's 8 threads (one fixed order)
            {
                const int cpr = I / 8, n = ncol * cpr;
#pragma unroll 1
                for (int b0 = 0; b0 < n; b0 += CT) {
                    const int idx = b0 + gt, c = idx / cpr, ch = idx - c * cpr;
                    uint4 hv = make_uint4(0u, 0u, 0u, 0u);
                    if (idx < n) {
                        hv = __ldcg(reinterpret_cast<const uint4 *>(a.h + (size_t)colf[c] * I) + ch);
                        *reinterpret_cast<uint4 *>(s_h + c * geo.h_stride + ch * 8) = hv;
                    }
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&hv.x));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&hv.y));
                    const float2 f2 = __half22float2(*reinterpret_cast<const __half2 *>(&hv.z));
                    const float2 f3 = __half22float2(*reinterpret_cast<const __half2 *>(&hv.w));
                    float sum = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
                    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                    if (idx < n && (ch & 7) == 0) s_hs[c * GI + (ch >> 3)] = sum;
                }
            }
            group_bar<CT>(gid);
            float acc[RT][NT][4];
#pragma unroll
            for (int t = 0; t < RT; ++t)
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[t][j][q] = 0.f;
            const int wrow = gw * 16 * RT;                          // first row of this warp in the unit
            const int ntile = min(RT, max(0, (H - rb * kRows2 - wrow) / 16));   // H is a multiple of 64
            const uint16_t *dsc = reinterpret_cast<const uint16_t *>(base + geo.sc2_off) + (wrow + g) * GI;
            const uint16_t *dbi = dsc + kRows2 * GI;
            const uint8_t *cb = base + (wrow + g) * 128;
            if (ntile > 0) {
                // one 128-byte code box (four groups) per step, unrolled; the h fragments serve every tile
#pragma unroll 1
                for (int bx = 0; bx < geo.nb2; ++bx) {
                    uint2 vs0[RT], vs1[RT], vb0[RT], vb1[RT];
#pragma unroll
                    for (int t = 0; t < RT; ++t) {
                        vs0[t] = lds_u2(dsc + (16 * t) * GI + 4 * bx);
                        vs1[t] = lds_u2(dsc + (16 * t + 8) * GI + 4 * bx);
                        vb0[t] = lds_u2(dbi + (16 * t) * GI + 4 * bx);
                        vb1[t] = lds_u2(dbi + (16 * t + 8) * GI + 4 * bx);
                    }
                    float4 hA[NT], hB[NT];                    // sums of h over the box's four groups
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const int cA = j * 8 + 2 * t4;
                        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                        hA[j] = cA < ncol ? *reinterpret_cast<const float4 *>(s_hs + cA * GI + 4 * bx) : z;
                        hB[j] = cA + 1 < ncol ? *reinterpret_cast<const float4 *>(s_hs + (cA + 1) * GI + 4 * bx) : z;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int grp = 4 * bx + q;
                        const uint32_t o = (uint32_t)bx * kBox2 + swz_chunk(q, g, t4);
                        uint32_t ad[RT][2][8];
#pragma unroll
                        for (int t = 0; t < RT; ++t) {
                            const uint2 c0 = *reinterpret_cast<const uint2 *>(cb + t * 2048 + o);
                            const uint2 c1 = *reinterpret_cast<const uint2 *>(cb + t * 2048 + o + 1024);
                            nib8<true>(c0.x, ad[t][0]);
                            nib8<true>(c0.y, ad[t][0] + 4);
                            nib8<true>(c1.x, ad[t][1]);
                            nib8<true>(c1.y, ad[t][1] + 4);
                        }
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            if (j * 8 >= ncol) break;
                            const int c = j * 8 + g;
                            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
                            if (c < ncol) {
                                const uint4 *hr =
                                    reinterpret_cast<const uint4 *>(s_h + c * geo.h_stride + grp * 64 + 16 * t4);
                                lo = hr[0];
                                hi = hr[1];
                            }
                            const float xA = f4_at(hA[j], q), xB = f4_at(hB[j], q);
#pragma unroll
                            for (int t = 0; t < RT; ++t) {
                                if (t >= ntile) break;
                                const float s0 = bf16x4_at(vs0[t], q), s1 = bf16x4_at(vs1[t], q);
                                const float k0 = fmaf(-1024.f, s0, bf16x4_at(vb0[t], q));
                                const float k1 = fmaf(-1024.f, s1, bf16x4_at(vb1[t], q));
                                float dd[4] = {0.f, 0.f, 0.f, 0.f};
                                mma16816<true>(dd, ad[t][0][0], ad[t][1][0], ad[t][0][1], ad[t][1][1], lo.x, lo.y);
                                mma16816<true>(dd, ad[t][0][2], ad[t][1][2], ad[t][0][3], ad[t][1][3], lo.z, lo.w);
                                mma16816<true>(dd, ad[t][0][4], ad[t][1][4], ad[t][0][5], ad[t][1][5], hi.x, hi.y);
                                mma16816<true>(dd, ad[t][0][6], ad[t][1][6], ad[t][0][7], ad[t][1][7], hi.z, hi.w);
                                acc[t][j][0] = fmaf(s0, dd[0], fmaf(k0, xA, acc[t][j][0]));
                                acc[t][j][1] = fmaf(s0, dd[1], fmaf(k0, xB, acc[t][j][1]));
                                acc[t][j][2] = fmaf(s1, dd[2], fmaf(k1, xA, acc[t][j][2]));
                                acc[t][j][3] = fmaf(s1, dd[3], fmaf(k1, xB, acc[t][j][3]));
                            }
                        }
                    }
                }
            }
            mbar_arrive_after(eb, acc[0][0][0], acc[0][0][2], acc[0][0][1], acc[0][0][3]);
#pragma unroll
            for (int t = 0; t < RT; ++t) {
                if (t >= ntile) break;
                const int w0 = rb * kRows2 + wrow + 16 * t + g, w1 = w0 + 8;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int cA = j * 8 + 2 * t4, cB = cA + 1;
                    if (cA < ncol) {
                        const int f = colf[cA];
                        a.yslot[(size_t)f * H + w0] = acc[t][j][0];
                        a.yslot[(size_t)f * H + w1] = acc[t][j][2];
                    }
                    if (cB < ncol) {
                        const int f = colf[cB];
                        a.yslot[(size_t)f * H + w0] = acc[t][j][1];
                        a.yslot[(size_t)f * H + w1] = acc[t][j][3];
                    }
                }
            }
            group_bar<CT>(gid);
            if (gt == 0) st_release_cta(&S.sig[gid], (i - gid) / CG + 1);
        }
    }
    if (CG > 1 && !past_gateup) all_consumers_bar();   // every consumer thread takes that barrier once
    // the remaining combines of this group, each as soon as the signal thread queues it, until it
    // has counted every unit (bounded)
#pragma unroll 1
    for (long long polls = 0;; ++polls) {
        if (gt == 0) {
            const int done = ld_acquire_cta(&S.sig_done);
            S.ncomb_snap[gid] = ld_acquire_cta(&S.ncomb);
            S.ready[gid] = done || polls > limit;
            if (!done && polls > limit) record_status(a.status, MOE_ERR_TIMEOUT);
        }
        group_bar<CT>(gid);
        const bool last = S.ready[gid];
        run_combines(S.ncomb_snap[gid]);
        if (last) break;
        if (gt == 0) __nanosleep(64);
        group_bar<CT>(gid);
    }
}

// ------------------------------------------------------------------ host side

// Consumer groups: two (alternating units) once a batch has more than two tokens, where a CTA
// has many units; one for one or two tokens, where each CTA has one or two units and all eight
// warps on a unit finish it soonest.
int consumer_groups(int T) { return T > 2 ? 2 : 1; }

// The ring layout needs 128-byte code boxes: H and I multiples of 256.
bool stream_geometry(int T, int H, int I, size_t smem_budget, StreamGeom *out)
{
    if (T < 1 || T > kDecodeMaxTok || H % 256 || I % 256 || H > 8192) return false;
    StreamGeom g{};
    const int G = H / kGroup, GI = I / kGroup, NT = T > 8 ? 2 : 1;
    g.nb1 = H / 256;
    g.up_off = (uint32_t)g.nb1 * kBox1;
    g.sc1_off = 2 * g.up_off;
    g.sb1 = (uint32_t)kRows1 * G * 2;
    g.bytes1 = 2 * g.up_off + 4 * g.sb1;
    const uint32_t size1 = g.sc1_off + 4 * g.sb1;
    g.nb2 = I / 256;
    g.sc2_off = (uint32_t)g.nb2 * kBox2;
    const uint32_t size2 = g.sc2_off + 2u * kRows2 * GI * 2;
    g.slot = (uint32_t)align_up(size1 > size2 ? size1 : size2, 1024);
    g.x_stride = H / 8 + 1;
    g.h_stride = I + 8;
    // x (read by the gate/up units) and each consumer group's staged h columns and their group
    // sums (read by the down units, which every CTA takes after all of its gate/up units) share
    // one region
    const size_t CG = consumer_groups(T);
    const size_t xb = (size_t)T * g.x_stride * 16, sumb = (size_t)T * G * 4;
    const size_t hb = CG * NT * 8 * g.h_stride * 2, hsb = CG * NT * 8 * GI * 4;
    const size_t region = std::max(align_up(xb, 16), align_up(hb, 16) + align_up(hsb, 16));
    const size_t redb = CG * kConsumerWarps * 2 * 16 * NT * 8 * 4;
    const size_t fixed = region + align_up(sumb, 16) + redb + 1024;
    const size_t budget = smem_budget - sizeof(SSmem) - 256;
    if (budget <= fixed) return false;
    size_t R = (budget - fixed) / g.slot;
    if (R > kMaxSlots) R = kMaxSlots;
    if (R < 2) return false;
    g.R = (int)R;
    size_t o = R * g.slot;
    g.x_off = g.h_off = (uint32_t)o;
    g.hs_off = (uint32_t)(o + align_up(hb, 16));
    o += region;
    g.sumx_off = (uint32_t)o;
    o += align_up(sumb, 16);
    g.red_off = (uint32_t)o;
    o += redb;
    g.dyn = (uint32_t)(o + 1024);      // slack for aligning the base to 1024 bytes
    *out = g;
    return true;
}

int dev_attr(int dev, cudaDeviceAttr attr, int slot)
{
    static int v[16][3] = {};
    int &r = v[dev & 15][slot];
    if (!r) cudaDeviceGetAttribute(&r, attr, dev);
    return r;
}
int optin_smem(int dev) { return dev_attr(dev, cudaDevAttrMaxSharedMemoryPerBlockOptin, 0); }
int sm_smem(int dev) { return dev_attr(dev, cudaDevAttrMaxSharedMemoryPerMultiprocessor, 1); }
int sm_count(int dev) { return dev_attr(dev, cudaDevAttrMultiProcessorCount, 2); }

// CTAs per SM and the matching geometry: two per SM when T <= 2 and half of the SM's
// shared memory still holds a ring of two slots (twice the warps on the few units
// of a one- or two-token batch), else one.
bool plan_launch(int T, int H, int I, int dev, StreamGeom *geo, int *per_sm)
{
    const size_t reserved = 1024;                  // per CTA, kept by the runtime
    if (T <= 2 && stream_geometry(T, H, I, (size_t)sm_smem(dev) / 2 - reserved, geo)) {
        *per_sm = 2;
        return true;
    }
    *per_sm = 1;
    return stream_geometry(T, H, I, (size_t)optin_smem(dev), geo);
}

// One copy per unit: the codes seen as (128-byte chunk, row, chunk index) with the chunk index
// outermost, so that the box lands in shared memory as the 2D boxes of the chunks one after the
// other (the 128-byte swizzle still keyed on the row).
bool code_map_whole(CUtensorMap *m, const uint8_t *codes, int row_bytes, uint64_t rows, int box_rows)
{
    const uint64_t dims[3] = {128u, rows, (uint64_t)row_bytes / 128u};
    const uint64_t strides[2] = {(uint64_t)row_bytes, 128u};
    const uint32_t box[3] = {128u, (uint32_t)box_rows, (uint32_t)row_bytes / 128u};
    return make_map_3d(m, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool code_map(CUtensorMap *m, const uint8_t *codes, int row_bytes, uint64_t rows, int box_rows)
{
    return make_map_2d(m, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)row_bytes, rows, 128u, (uint32_t)box_rows,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool decode_stream_fits(int T, int H, int I)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    StreamGeom g;
    int per_sm = 0;
    return plan_launch(T, H, I, dev, &g, &per_sm);
}

cudaError_t launch_decode_stream(const FusedDecodeArgs &a, cudaStream_t st)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    StreamGeom geo;
    int want = 1;
    if (!plan_launch(a.T, a.H, a.I, dev, &geo, &want)) return cudaErrorInvalidValue;
    StreamMaps maps;
    const uint64_t E = (uint64_t)a.E;
    // whole-unit 3D maps where the driver takes them, else one 2D map box per 128-byte chunk
    bool ok = false;
    for (int whole = 1; whole >= 0 && !ok; --whole) {
        auto mk = whole ? code_map_whole : code_map;
        maps.whole = whole;
        ok = mk(&maps.g, a.gate.codes, a.H / 2, E * a.I, kRows1) && mk(&maps.u, a.up.codes, a.H / 2, E * a.I, kRows1) &&
             mk(&maps.d, a.down.codes, a.I / 2, E * a.H, kRows2);
        if (ok && a.has_shared)
            ok = mk(&maps.sg, a.s_gate.codes, a.H / 2, a.I, kRows1) && mk(&maps.su, a.s_up.codes, a.H / 2, a.I, kRows1) &&
                 mk(&maps.sd, a.s_down.codes, a.I / 2, a.H, kRows2);
        else if (ok) {
            maps.sg = maps.g;
            maps.su = maps.u;
            maps.sd = maps.d;
        }
    }
    if (!ok) return cudaErrorInvalidValue;
    auto kern = a.T > 8                      ? decode_stream_kernel<2, 1, 2>
                : consumer_groups(a.T) == 2  ? decode_stream_kernel<1, 1, 2>
                : want == 2                  ? decode_stream_kernel<1, 2, 1>
                                             : decode_stream_kernel<1, 1, 1>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.dyn)) != cudaSuccess)
        return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSThreads, geo.dyn)) != cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count(dev) * (per_sm < want ? per_sm : want));
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = geo.dyn;
    cfg.stream = st;
    // cooperative (the CTAs wait on one another), and allowed to start while the router
    // kernel before it still runs: phase 0 waits for it after staging x
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, maps, a, geo);
}

}  // namespace qmoe
