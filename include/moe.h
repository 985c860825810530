/*
 * moe.h - C ABI of the GB300 (sm_103a) routed-expert MoE layer library (libmoe.so).
 *
 * The layer is the qwen3_5_moe routed-expert MLP with the routing and combine
 * contract set out on the page "Qwen3.6-35B-A3B (qwen3_5_moe) on the native
 * Metal engine: proposal and gate", section "What I'd build, in slices",
 * slice "The family, plain decode":
 *   1. fp32 router logits over the E experts, and the shared expert's fp32 gate
 *      logit gamma = x . v;
 *   2. top-k experts by logit, ties going to the lower expert id;
 *   3. pick weights exp(l - l_top) over the k picks, normalised over the picks
 *      (the "softmax top-8" of the "Qwen-3.6-35B-A3B-SIQ-K6-K4K3" model card,
 *      section "Reproduction"), rounded to bf16;
 *   4. the shared expert is one more slot with weight bf16(sigmoid(bf16(gamma)));
 *   5. each expert is a SwiGLU MLP, y_e = W_down (silu(W_gate x) * (W_up x))
 *      (the Gate section's "expert gate/up pair, expert down");
 *   6. y = bf16( sum_j p_j y_{e_j} + w_s y_shared ), rounded once.
 * Weights are MLX affine quantised (same slice): experts 4-bit, router 8-bit,
 * groups of 64 consecutive inputs of one output row sharing a bf16 scale s
 * and bias b, w = s * q + b.  The page's slice "8-bit experts" (the same
 * rule with expert codes q in [0, 255]) is supported too: moe_config.bits = 8.
 * Code layout: a row of n inputs holds n * bits / 8 bytes; at 4 bits input j
 * is the low nibble of byte j / 2 for even j and the high nibble for odd j,
 * at 8 bits input j is byte j.
 * Block-scaled experts (moe_config.format = MOE_FORMAT_NVFP4): every expert
 * matrix, shared included, in NVFP4, the checkpoint format named on the model
 * card "Qwen-3.6-35B-A3B-SIQ-K6-K4K3" (served there by a fused FP4 MoE
 * backend); the router stays 8-bit affine.  w_j = e2m1(q_j) * e4m3(s_b) * g
 * with q_j a 4-bit E2M1 code (bit 3 sign, bits 2..1 exponent with bias 1,
 * bit 0 mantissa; packed as the 4-bit affine codes), s_b the E4M3 scale of
 * the block of 16 consecutive inputs holding j, g the matrix's fp32 scale.
 *
 * Conventions shared by every entry point
 *   - Every function returns an int status (enum moe_status).  Argument,
 *     shape and format errors are found on the host, before anything is
 *     enqueued, and leave every buffer untouched.
 *   - Pointers to tensors are caller-owned DEVICE memory unless a parameter
 *     says otherwise.  The library never allocates, frees or synchronises,
 *     except moe_get_device_status, which synchronises the given stream.
 *   - Every tensor pointer must be 16-byte aligned; rows are dense (no
 *     padding between rows).  bf16 tensors are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All work is enqueued asynchronously on it, in order.
 *   - `ws`/`ws_bytes` is caller-owned device scratch of at least
 *     moe_workspace_size() bytes for the call's T; it must not be shared by
 *     calls that may run concurrently.  Its first 512 bytes (the header: the
 *     status word and the grid-wide counters of the fused decode kernel) must
 *     be zero before the workspace's first use: allocate it zero-filled, or
 *     call moe_get_device_status on it once.  The kernels leave the counters
 *     zero when they end; the rest of the workspace carries nothing between
 *     calls.  A header that was not zero-filled is detected as far as the
 *     kernels can (MOE_ERR_WORKSPACE in the status word).
 *   - Device-side failures (a bounded wait that ran out, an index out of
 *     range, a header that was not zero-filled) never trap: the kernel writes
 *     a nonzero code into the workspace status word and returns.  The word
 *     keeps the first such code until moe_get_device_status reads it.
 *   - Values: x and the weights are finite.  Each token's x is scaled by a
 *     power of two before the 16-bit intermediate steps and the scale is
 *     undone after them (exact), so rows far above the fp16 range or entirely
 *     below its normal range keep their precision (within a row, elements
 *     below 2^-17 of its largest are held to fp16's subnormal spacing, an
 *     error of at most 2^-25 of that largest); only an output beyond the
 *     bf16 range overflows.
 *
 * Storage formats (MLX layout, [out, in] with quantisation along `in`)
 *   codes   4-bit: uint8 [rows, in/2], element j of a row in byte j/2, low
 *           nibble for even j.  8-bit: uint8 [rows, in].
 *   scales, biases: bf16 [rows, in/group].
 *   NVFP4 experts: codes as the 4-bit codes; scales holds E4M3 bytes
 *           [rows, in/16] (passed through the scales pointer); biases unused
 *           (may be NULL); gscale fp32, one per matrix ([E] for a stack).
 *           A NaN scale code (0x7F, 0xFF) makes the rows it scales undefined.
 *   Stacked expert matrices add a leading expert dimension:
 *     gate, up   [E, inter, hidden]     down  [E, hidden, inter]
 *     s_gate, s_up [inter, hidden]      s_down [hidden, inter]   (shared expert)
 *     router     [E, hidden] (8-bit)    shared_gate_vec bf16 [hidden]
 */
#ifndef QMOE_GB300_MOE_H
#define QMOE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, negative or oversized size */
    MOE_ERR_UNSUPPORTED = 2,  /* a format or shape the kernels do not implement */
    MOE_ERR_WORKSPACE = 3,    /* ws_bytes below moe_workspace_size(); as a device status: a
                                 workspace header that was not zero-filled */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, attribute query) */
    MOE_ERR_TIMEOUT = 5,      /* device status: a bounded wait inside a kernel ran out */
    MOE_ERR_DEVICE = 6        /* device status: a kernel found an index out of range */
};

enum moe_path {
    MOE_PATH_AUTO = 0,     /* decode for T <= 16, prefill above */
    MOE_PATH_DECODE = 1,   /* weight-streaming dequant-GEMV kernels (any T, meant for small T) */
    MOE_PATH_PREFILL = 2   /* tcgen05 grouped GEMM kernels (any T >= 1) */
};

/* Layer shape and per-call options.  Supported: group == 64, bits == 4 or 8
 * (4 with format == MOE_FORMAT_NVFP4), router_bits == 8, hidden and inter multiples of 64 (hidden <= 8192,
 * inter <= 4096), 1 <= top_k <= min(n_experts, 16), 1 <= n_experts <= 256,
 * has_shared in {0,1}.  Anything else returns MOE_ERR_UNSUPPORTED.
 * wait_polls bounds the in-kernel waits of the call: a wait polls at most
 * that many times (the first poll does not block, later ones sleep briefly),
 * then records MOE_ERR_TIMEOUT and the kernel returns early.  0 (or less)
 * selects the default, 1 << 20 polls (about a second).  A limit of 1 makes
 * any such wait that is not already satisfied run out (fault tests).  In the
 * fused decode kernel (T <= 16) it bounds the waits on other CTAs (published
 * router logits, the grid-wide unit counter); a CTA's waits on its own
 * shared-memory copies keep a fixed bound of the same order, so that a small
 * limit never leaves the copy ring in mid-flight.
 * With bits == 8 the decode path runs the weight-streaming gate/up, down and
 * reduce kernels after the routing kernels (the fused decode kernel and the
 * packed down layout are for 4-bit affine codes), and the prefill path runs
 * every expert on the tensor-memory GEMMs.  NVFP4 experts take the prefill
 * path at every T (MOE_PATH_DECODE and MOE_PATH_AUTO select it too). */
/* Expert storage formats (moe_config.format). */
enum moe_format {
    MOE_FORMAT_AFFINE = 0,  /* MLX affine, bits 4 or 8, groups of 64 */
    MOE_FORMAT_NVFP4 = 1    /* E2M1 codes, E4M3 scale per 16 inputs, fp32 per matrix; bits == 4 */
};

typedef struct moe_config {
    int hidden;       /* H */
    int inter;        /* I, intermediate size of every expert, shared included */
    int n_experts;    /* E routed experts */
    int top_k;        /* k picks per token */
    int group;        /* quantisation group along the input dimension */
    int bits;         /* expert code width */
    int router_bits;  /* router code width */
    int has_shared;   /* 1: the layer has a shared expert slot */
    int wait_polls;   /* bound on the in-kernel waits of the call; 0 = default */
    int format;       /* expert storage format, enum moe_format (0 = affine) */
} moe_config;

/* One quantised matrix (or a stack of them), device pointers, 16-byte aligned
 * (gscale: 4-byte aligned). */
typedef struct moe_qmat {
    const uint8_t *codes;
    const uint16_t *scales;  /* affine: bf16; NVFP4: E4M3 bytes */
    const uint16_t *biases;  /* affine: bf16; NVFP4: unused */
    const float *gscale;     /* NVFP4: fp32 scale per matrix; affine: unused */
} moe_qmat;

/* All weights of one layer, device pointers.  s_* and shared_gate_vec may be
 * NULL when has_shared == 0.
 * down_packed / s_down_packed (optional, NULL for none): the down codes
 * rearranged by moe_pack_down, which the decode kernel streams one contiguous
 * block per (expert, 32 columns of the intermediate dimension) instead of
 * gathering 16-byte pieces of every row.  They are read only by the decode
 * path and give the same results as the MLX layout. */
typedef struct moe_weights {
    moe_qmat router;   /* [E, H], router_bits */
    moe_qmat gate;     /* [E, I, H] */
    moe_qmat up;       /* [E, I, H] */
    moe_qmat down;     /* [E, H, I] */
    moe_qmat s_gate;   /* [I, H] */
    moe_qmat s_up;     /* [I, H] */
    moe_qmat s_down;   /* [H, I] */
    const uint16_t *shared_gate_vec;  /* bf16 [H] */
    const uint8_t *down_packed;       /* [E, I/32, H, 16] bytes, or NULL */
    const uint8_t *s_down_packed;     /* [I/32, H, 16] bytes, or NULL */
} moe_weights;

/* Human-readable name of a status code; never NULL, static storage. */
MOE_API const char *moe_status_string(int status);

/* Checks a configuration against the supported set (see moe_config). */
MOE_API int moe_check_config(const moe_config *cfg);

/* Bytes of workspace every entry point below needs for T tokens (0 <= T <= 65536).
 * *bytes receives the size; the same workspace serves every entry point. */
MOE_API int moe_workspace_size(const moe_config *cfg, int T, size_t *bytes);

/* Steps 1-4: router logits, top-k, pick weights, shared weight.
 *   x           bf16 [T, H]
 *   router_bias fp32 [E] added to every computed logit with one fp32 rounding
 *               (l = fp32(l + bias_e)); NULL for none.  Ignored with logits_in.
 *   logits_in   fp32 [T, E] logits to route on instead of the router GEMV; NULL
 *               to compute them.  Lets a caller with its own router use the layer.
 *   logits_out  fp32 [T, E] or NULL: the logits the top-k ran on.
 *   ids         int32 [T, k] expert ids in rank order (descending logit, ties
 *               to the lower id).
 *   p           bf16 [T, k] pick weights in the same order.
 *   w_shared    bf16 [T] shared-slot weight; NULL allowed; all zero when
 *               has_shared == 0.
 * T == 0 is valid and enqueues nothing. */
MOE_API int moe_route(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int T,
              const float *router_bias, const float *logits_in, float *logits_out,
              int32_t *ids, uint16_t *p, uint16_t *w_shared,
              void *ws, size_t ws_bytes, void *stream);

/* Groups the T*k routed slots by expert: a stable counting sort of the flat
 * slot index f = t*k + j by ids[f] (so slots of one expert are in increasing t).
 *   counts   int32 [E]      slots routed to each expert
 *   offsets  int32 [E + 1]  exclusive prefix sum of counts
 *   perm     int32 [T*k]    perm[offsets[e] + r] = r-th slot routed to e
 *   inv_perm int32 [T*k]    inv_perm[f] = position of slot f in perm
 * ids entries outside [0, E) set MOE_ERR_DEVICE in the status word and the
 * outputs are then unspecified. */
MOE_API int moe_permute(const moe_config *cfg, const int32_t *ids, int T, int32_t *counts,
                int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                void *ws, size_t ws_bytes, void *stream);

/* Step 5 and the weighted sum of step 6 without its rounding:
 *   acc[t, :] += sum_j p[t,j] * y_{ids[t,j]}(x_t) + w_shared[t] * y_shared(x_t)
 * acc is fp32 [T, H], caller-initialised (zero for a plain layer).
 * ids/p/w_shared as produced by moe_route; counts/offsets/perm as produced by
 * moe_permute from the same ids.  w_shared may be NULL when has_shared == 0.
 * path selects the kernels (enum moe_path).  On both paths each slot's expert
 * output is computed once and every acc element receives one fixed-order sum
 * of them, so the result is bit-reproducible for a given batch.  On the decode
 * path it is also independent of the other tokens in the batch; on the
 * prefill path an expert's token count selects the kernels that compute it
 * (exact-code small tiles up to 32 tokens, fp16-dequantised tensor-memory
 * GEMMs above), so a token's last bits can depend on its batch. */
MOE_API int moe_expert_ffn(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int T,
                   const int32_t *ids, const uint16_t *p, const uint16_t *w_shared,
                   const int32_t *counts, const int32_t *offsets, const int32_t *perm,
                   float *acc, int path, void *ws, size_t ws_bytes, void *stream);

/* The single rounding of step 6: y = bf16_rne(acc), acc fp32 [T, H], y bf16 [T, H]. */
MOE_API int moe_combine(const moe_config *cfg, int T, const float *acc, uint16_t *y, void *stream);

/* The whole layer: route, permute, expert FFNs and combine.
 *   y        bf16 [T, H] output.
 *   ids_out  int32 [T, k], p_out bf16 [T, k], w_shared_out bf16 [T]: optional
 *            copies of the routing (NULL to skip).
 * Other arguments as in moe_route / moe_expert_ffn.  With MOE_PATH_DECODE
 * (or AUTO with T <= 16) row t of y, ids_out, p_out and w_shared_out is
 * bit-identical to the result of a T = 1 call on row t alone. */
MOE_API int moe_forward(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int T,
                const float *router_bias, const float *logits_in, uint16_t *y,
                int32_t *ids_out, uint16_t *p_out, uint16_t *w_shared_out, int path,
                void *ws, size_t ws_bytes, void *stream);

/* The decode layer (T <= 16) for callers that cannot allocate device memory.
 * The pages describe nothing like it: it exists for callers such as code that
 * runs inside another engine's enqueue callback (that engine owns all device
 * memory) or a process that must not allocate after start-up.
 * Same arguments and results as moe_forward with MOE_PATH_DECODE, but no
 * workspace: the scratch is a fixed 24 MiB array in the library's own device
 * memory, held on every GPU that loads the library until the process exits
 * (zero at load; the kernels leave its counters zero).  Layers whose decode
 * scratch exceeds 24 MiB are refused with MOE_ERR_WORKSPACE; T outside 0..16
 * with MOE_ERR_INVALID_ARG.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array, which keeps the last call's
 * contents: calls that overlap on the GPU (other streams, other threads)
 * race and give wrong results, so keep them ordered.  Device-side status is
 * recorded in the array and cannot be read back.  Allocates nothing. */
MOE_API int moe_forward_decode_static(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int T,
                                      const float *router_bias, const float *logits_in, uint16_t *y,
                                      int32_t *ids_out, uint16_t *p_out, uint16_t *w_shared_out, void *stream);

/* Writes the decode layout of the 4-bit down codes (bits == 4 only, else
 * MOE_ERR_UNSUPPORTED): for expert e and column
 * slice c (32 columns of the intermediate dimension, 16 bytes of every row),
 *   down_packed[((e * (I/32) + c) * H + r) * 16 + b] = down.codes[(e * H + r) * I/2 + c * 16 + b]
 * and the same for the shared expert into s_down_packed (skipped when NULL or
 * has_shared == 0).  Each output holds as many bytes as its source; both are
 * caller-owned device memory.  Enqueued on `stream`; run it once after the
 * weights are loaded. */
MOE_API int moe_pack_down(const moe_config *cfg, const moe_weights *w, uint8_t *down_packed,
                          uint8_t *s_down_packed, void *stream);

/* Synchronises `stream`, then reads the device status word of `ws` and zeroes
 * the workspace header (status word and counters).  *device_status receives
 * MOE_OK or the first error code a kernel recorded since the last read. */
MOE_API int moe_get_device_status(void *ws, size_t ws_bytes, void *stream, int *device_status);

/* The intermediate stages of the expert FFNs, for checking each projection on
 * its own (the FP64 check of every projection class in the section "Gate" of
 * the proposal page): for every slot f (routed: f = t k + j, shared:
 * f = T k + t)
 *   h_out     fp32 [T (k + 1), I]  h = silu(W_gate x) * (W_up x) exactly as the
 *             down projection consumes it (after the kernels' own rounding), or NULL;
 *   yslot_out fp32 [T (k + 1), H]  the slot's expert output W_down h before the
 *             pick weight, or NULL.
 * ids/counts/offsets/perm as for moe_expert_ffn (counts/offsets/perm are read
 * on the prefill path only).  The same kernels as moe_expert_ffn compute the
 * stages; nothing is added into an accumulator.  Rows of h_out / yslot_out
 * of slots that do not exist (the
 * shared rows without a shared expert) are not written.  Returns
 * MOE_ERR_UNSUPPORTED for a path whose kernels cannot emit their stages (the
 * decode path of a layer that does not take the fused decode kernel: bits == 8,
 * or a shape outside its shared-memory plan). */
MOE_API int moe_expert_stages(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int T,
                              const int32_t *ids, const int32_t *counts, const int32_t *offsets,
                              const int32_t *perm, float *h_out, float *yslot_out, int path,
                              void *ws, size_t ws_bytes, void *stream);

/* Timeline of the last fused decode launch on `ws` (T <= 16, decode path):
 * synchronises `stream`, then copies per CTA fourteen %globaltimer stamps
 * (ns) to host_stamps [max_ctas, 14]: kernel start, router logits published,
 * every logit seen, x staged for the expert units, top-k done, expert list
 * done, routing done, first gate chunk landed, first down chunk landed, first
 * down chunk computed, expert units done, unit counter reached, combine loads
 * done, combine done (a stamp that was not reached keeps an older value).
 * *n_ctas receives the number of CTAs of the launch. */
MOE_API int moe_decode_timeline(const moe_config *cfg, int T, void *ws, size_t ws_bytes, void *stream,
                                unsigned long long *host_stamps, int max_ctas, int *n_ctas);

#ifdef __cplusplus
}
#endif
#endif /* QMOE_GB300_MOE_H */
