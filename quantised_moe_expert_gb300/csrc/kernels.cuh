// Kernel argument blocks and launchers of the MoE layer library.
#pragma once

#include "moe_common.cuh"

namespace qmoe {

struct RouteArgs {
    const uint16_t *x;            // bf16 [T, H]
    const uint8_t *r_codes;       // u8 [E, H]
    const uint16_t *r_scales;     // bf16 [E, H/64]
    const uint16_t *r_biases;
    const uint16_t *v;            // bf16 [H] shared gate vector (may be null)
    const float *router_bias;     // f32 [E] or null
    float *logits;                // f32 [T, E]
    float *gamma;                 // f32 [T]
    int *status_reset;            // non-null: cleared by the first thread (first kernel of a call)
    int *zero;                    // non-null: block (0,0) zeroes zero[0, nzero) (counters of the next kernel)
    int nzero;
    int T, H, E;
    int n_expert_tiles;           // 0: only the gamma column runs
};

struct RouterMmaArgs {
    const uint16_t *x;            // bf16 [T, H]
    const uint8_t *codes;         // u8 [E, H]
    const uint16_t *scales;       // bf16 [E, H/64]
    const uint16_t *biases;
    const float *router_bias;     // f32 [E] or null
    float *logits;                // f32 [T, E]
    int T, H, E;
};

cudaError_t launch_router_mma(const RouterMmaArgs &a, cudaStream_t st);

struct TopkArgs {
    const float *logits;          // f32 [T, E]
    const float *gamma;           // f32 [T]
    int32_t *ids;                 // [T, k]
    uint16_t *p;                  // bf16 [T, k]
    uint16_t *w_s;                // bf16 [T] (may be null)
    int32_t *hist;                // [nblk, E], zeroed beforehand; slots of tokens [128 b, 128 b + 128) count into row b
    int T, E, k, has_shared;
};

struct PermuteArgs {
    const int32_t *ids;
    const int32_t *hist;
    int32_t *counts, *offsets, *perm, *inv_perm;
    int32_t *nwork;               // [5]: decode items, gemm1 items, gemm2 items, gemm1 / gemm2 items of the big kernels
    WorkItem *work_dec, *work_g1, *work_g2;
    int *status;
    int T, E, k, nblk, has_shared;
    int build_work;               // block 0 also writes the expert kernels' work lists
    int small_tiles;              // GEMM lists split for the small-tile kernels
    int max_items[3];             // capacity of each work list
};

struct HistArgs {
    const int32_t *ids;
    int32_t *hist;
    int *status;
    int T, E, k, nblk;
};

struct WorklistArgs {
    const int32_t *counts;
    int32_t *nwork;
    WorkItem *work_dec, *work_g1, *work_g2;
    int *status;
    int *zero;                    // non-null: zero[0, nzero) (counters of the fused decode kernel)
    int nzero;
    int T, E, has_shared;
    int small_tiles;              // GEMM lists split for the small-tile kernels
    int max_items[3];
};

// One expert matrix stack as the expert kernels see it.
struct QMatDev {
    const uint8_t *codes;
    const uint16_t *scales;       // NVFP4: E4M3 block scales, read as bytes
    const uint16_t *biases;
    const float *gscale;          // NVFP4: fp32 scale per matrix
};

// Value of the args' `bits` field for NVFP4 experts (4-bit E2M1 codes, E4M3 scale per 16 inputs,
// fp32 scale per matrix); 4 and 8 are the affine code widths.
constexpr int kNvfp4 = 5;

struct ExpertArgs {
    const uint16_t *x;            // bf16 [T, H]
    QMatDev gate, up, down;       // stacked [E, ...]
    QMatDev s_gate, s_up, s_down; // shared expert
    const int32_t *offsets;       // [E + 1]
    const int32_t *perm;          // [T*k]
    const int32_t *nwork;         // [3]
    const WorkItem *work;         // decode items or GEMM tiles
    uint16_t *h;                  // fp16 [T*k + T, I], slot-major (f = t*k + j; shared f = T*k + t): h 2^-2e
    float *yslot;                 // f32 [T*k + T, H] (decode)
    int *xe;                      // i32 [T]: e of each token, 2^e <= max |x| < 2^(e + 1) (workspace)
    const uint16_t *p;            // bf16 [T, k]
    const uint16_t *w_s;          // bf16 [T]
    float *acc;                   // f32 [T, H]
    int *status;
    int T, H, I, E, k, has_shared;
    int bits;                     // expert codes: 4 or 8 (affine), kNvfp4
    int max_items;
};

struct ReduceArgs {
    const float *yslot;           // f32 [T (k + 1), H] slot outputs
    const int32_t *pos;           // [T k] row of yslot holding routed slot f (null: row f); shared slot T k + t: row T k + t
    int *status;
    const uint16_t *p;
    const uint16_t *w_s;
    float *acc;                   // acc += sum (when y == null)
    uint16_t *y;                  // y = bf16(sum) (when non-null)
    int T, H, k, has_shared;
};

struct PrefillArgs {
    const uint16_t *x;            // bf16 [T, H]
    uint16_t *x16;                // fp16 [T, H] scratch (K-permuted): x' = x 2^-e per token
    float *xsum;                  // f32 [T, H / 64] scratch: group sums of x16
    int *xe;                      // i32 [T] scratch: the token's e (max |x'| in [1, 2))
    float *hsum;                  // f32 [T*k + T, I / 64] scratch: group sums of h (small-tile items)
    uint16_t *hs;                 // fp16 [T*k + T, I] scratch, expert-sorted rows
    QMatDev gate, up, down, s_gate, s_up, s_down;
    const int32_t *nwork, *offsets, *perm;
    const WorkItem *work_g1, *work_g2;
    float *h_out;                 // f32 [T (k + 1), I] h per slot (stage output), or null
    float *yslot;                 // f32 [T (k + 1), H] each slot's expert output before its pick weight, rows in
                                  // expert-sorted position order (every element of the slots present written once)
    int *status;
    int T, H, I, E, k, has_shared, max_w1, max_w2;
    int bits;                     // expert codes: 4 or 8 (affine), kNvfp4
    long long wait_limit;
};

cudaError_t launch_prefill_experts(const PrefillArgs &a, cudaStream_t st);

// Small-tile grouped GEMMs (items of at most kSmallN tokens, exact int4 codes on mma.sync):
// whether a layer shape takes them (4-bit experts only), and their launches (items
// [nwork[3], nwork[1]) of the gate/up list, [nwork[4], nwork[2]) of the down list).
bool prefill_small_fits(int H, int I, int bits);
cudaError_t launch_small_gateup(const PrefillArgs &a, cudaStream_t st);
cudaError_t launch_small_down(const PrefillArgs &a, cudaStream_t st);

struct FusedDecodeArgs {
    const uint16_t *x;            // bf16 [T, H]
    const uint8_t *r_codes;       // router u8 [E, H]
    const uint16_t *r_scales;     // bf16 [E, H/64]
    const uint16_t *r_biases;
    const uint16_t *v;            // bf16 [H] shared gate vector (null without a shared expert)
    const float *router_bias;     // f32 [E] or null
    const float *logits_in;       // f32 [T, E] caller logits (no router GEMV), or null
    QMatDev gate, up, down, s_gate, s_up, s_down;
    const uint8_t *down_packed;   // down codes in the slice layout [E, I/32, H, 16], or null (gathered)
    const uint8_t *s_down_packed; // shared expert, [I/32, H, 16], or null
    const int32_t *ids_in;        // [T, k] given routing (then p_in / ws_in too), or null
    const uint16_t *p_in;         // bf16 [T, k]
    const uint16_t *ws_in;        // bf16 [T] or null
    int32_t *ids_out;             // [T, k] or null
    uint16_t *p_out;              // bf16 [T, k] or null
    uint16_t *ws_out;             // bf16 [T] or null
    unsigned long long *logits64; // [T, E] published logits: fp32 bits | epoch << 32 (workspace)
    uint16_t *p_glob;             // bf16 [T, k] published pick weights (workspace)
    uint16_t *ws_glob;            // bf16 [T] published shared weights (workspace)
    float *part;                  // f32 [T (k + 1), I / 32, H] raw down sums per column and slice (workspace)
    float *hsum;                  // f32 [T (k + 1), I / 32] sums of h' per column and slice (workspace)
    uint16_t *y;                  // bf16 [T, H] = bf16(sum), or null
    float *acc;                   // f32 [T, H] += sum (when y is null)
    float *h_out;                 // f32 [T (k + 1), I] h per slot as the down projection consumes it, or null
    float *yslot_out;             // f32 [T (k + 1), H] expert output per slot before weighting, or null
    int stages_only;              // 1: write h_out / yslot_out only (no y, no acc)
    int *sync;                    // workspace header: status word, then the three counters
    int *status;
    unsigned long long *trace;    // [grid, kTraceStamps] %globaltimer stamps per CTA, or null
    int T, H, I, E, k, has_shared;
    long long wait_limit;
};

// Fused decode kernel (T <= 16): router, top-k, expert FFNs and combine in one cooperative
// launch of one CTA per SM.  decode_fused_fits: whether the layer shape fits its shared-memory
// plan on the current device; decode_fused_trace_ctas: CTAs of that launch (rows of the trace).
bool decode_fused_fits(int T, int H, int I, int E, int k, int has_shared);
size_t decode_fused_trace_ctas();
cudaError_t launch_decode_fused(const FusedDecodeArgs &a, cudaStream_t st);
// Down codes [n, H, I/2] -> slice layout [n, I/32, H, 16].
cudaError_t launch_pack_down(const uint8_t *src, uint8_t *dst, int n, int H, int I, cudaStream_t st);
cudaError_t launch_route_gemv(const RouteArgs &a, cudaStream_t st);
cudaError_t launch_topk(const TopkArgs &a, cudaStream_t st);
cudaError_t launch_permute(const PermuteArgs &a, cudaStream_t st);
cudaError_t launch_hist(const HistArgs &a, cudaStream_t st);
cudaError_t launch_worklist(const WorklistArgs &a, cudaStream_t st);
cudaError_t launch_decode_gateup(const ExpertArgs &a, cudaStream_t st);
cudaError_t launch_decode_down(const ExpertArgs &a, cudaStream_t st);
// y (or acc) from the slot outputs: the fixed-order weighted sum over each token's slots.
cudaError_t launch_slot_sum(const ReduceArgs &a, cudaStream_t st);
// inv[perm[i]] = i for i < n (an entry out of range is reported in status and skipped).
cudaError_t launch_invert_perm(const int32_t *perm, int32_t *inv, int n, int *status, cudaStream_t st);
// out[f, :] = yslot[pos[f], :] for routed slots f < T k, out[f, :] = yslot[f, :] for shared slots.
cudaError_t launch_slot_gather(const float *yslot, const int32_t *pos, float *out, int T, int H, int k, int has_shared,
                               int *status, cudaStream_t st);
cudaError_t launch_combine(const float *acc, uint16_t *y, size_t n, cudaStream_t st);

}  // namespace qmoe
