// C ABI of the MoE layer library: argument checks, workspace carving, launches.
// The operations and their contract are stated in include/moe.h.
#include "kernels.cuh"

using namespace qmoe;

namespace {

constexpr long long kDefaultWaitPolls = 1ll << 20;

// Polls of every bounded wait inside the kernels of one call (moe_config.wait_polls).
long long wait_limit_of(const moe_config &c) { return c.wait_polls > 0 ? (long long)c.wait_polls : kDefaultWaitPolls; }

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned16_or_null(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool qmat_ok(const moe_qmat &m, bool nvfp4 = false)
{
    if (nvfp4)
        return aligned16(m.codes) && aligned16(m.scales) && m.gscale &&
               (reinterpret_cast<uintptr_t>(m.gscale) & 3u) == 0;
    return aligned16(m.codes) && aligned16(m.scales) && aligned16(m.biases);
}

// The args' code field: the affine code width, or kNvfp4.
int qcode(const moe_config &c) { return c.format == MOE_FORMAT_NVFP4 ? kNvfp4 : c.bits; }

template <typename T>
T *ws_at(void *ws, size_t off) { return reinterpret_cast<T *>(static_cast<char *>(ws) + off); }

QMatDev dev(const moe_qmat &m) { return QMatDev{m.codes, m.scales, m.biases, m.gscale}; }

int check_common(const moe_config *cfg, int T)
{
    if (!cfg) return MOE_ERR_INVALID_ARG;
    const int rc = moe_check_config(cfg);
    if (rc != MOE_OK) return rc;
    if (T < 0 || T > kMaxTokens) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

int check_ws(const moe_config *cfg, int T, void *ws, size_t ws_bytes, WsLayout *L)
{
    *L = ws_layout(*cfg, T);
    if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < L->total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// NVFP4 experts run on the tensor-memory GEMMs at every T (the weight-streaming decode kernels take
// affine codes).
int resolve_path(const moe_config &c, int path, int T)
{
    if (c.format == MOE_FORMAT_NVFP4) return MOE_PATH_PREFILL;
    if (path == MOE_PATH_AUTO) return T <= kDecodeMaxTok ? MOE_PATH_DECODE : MOE_PATH_PREFILL;
    return path;
}

// Arguments of the router GEMV kernel (logits and gamma).
RouteArgs route_args(const moe_config &c, const moe_weights &w, const uint16_t *x, int T, const float *router_bias,
                     const float *logits_in, float *logits, const WsLayout &L, void *ws)
{
    RouteArgs ra{};
    ra.x = x;
    ra.r_codes = w.router.codes;
    ra.r_scales = w.router.scales;
    ra.r_biases = w.router.biases;
    ra.v = c.has_shared ? w.shared_gate_vec : nullptr;
    ra.router_bias = router_bias;
    ra.logits = logits;
    ra.gamma = ws_at<float>(ws, L.gamma);
    ra.status_reset = nullptr;        // the status word keeps the first error until it is read
    ra.T = T;
    ra.H = c.hidden;
    ra.E = c.n_experts;
    ra.n_expert_tiles = logits_in ? 0 : (c.n_experts + 7) / 8;
    return ra;
}

int enqueue_route(const moe_config &c, const moe_weights &w, const uint16_t *x, int T, const float *router_bias,
                  const float *logits_in, float *logits, int32_t *ids, uint16_t *p, uint16_t *w_s,
                  const WsLayout &L, void *ws, cudaStream_t st)
{
    RouteArgs ra = route_args(c, w, x, T, router_bias, logits_in, logits, L, ws);
    const bool mma_router = !logits_in && T > kDecodeMaxTok;
    if (mma_router) ra.n_expert_tiles = 0;                  // gamma (and the histogram zeroing) only
    ra.zero = ws_at<int>(ws, L.hist);                       // the top-k counts into a zeroed histogram
    ra.nzero = L.nblk * c.n_experts;
    int rc = cuda_rc(launch_route_gemv(ra, st));
    if (rc) return rc;
    if (mma_router) {
        RouterMmaArgs rm{};
        rm.x = x;
        rm.codes = w.router.codes;
        rm.scales = w.router.scales;
        rm.biases = w.router.biases;
        rm.router_bias = router_bias;
        rm.logits = logits;
        rm.T = T;
        rm.H = c.hidden;
        rm.E = c.n_experts;
        if ((rc = cuda_rc(launch_router_mma(rm, st)))) return rc;
    }
    if (logits_in && logits && logits != logits_in) {
        rc = cuda_rc(cudaMemcpyAsync(logits, logits_in, sizeof(float) * (size_t)T * c.n_experts,
                                     cudaMemcpyDeviceToDevice, st));
        if (rc) return rc;
    }
    TopkArgs ta{};
    ta.logits = logits_in ? logits_in : logits;
    ta.gamma = ra.gamma;
    ta.ids = ids;
    ta.p = p;
    ta.w_s = w_s;
    ta.hist = ws_at<int32_t>(ws, L.hist);
    ta.T = T;
    ta.E = c.n_experts;
    ta.k = c.top_k;
    ta.has_shared = c.has_shared;
    return cuda_rc(launch_topk(ta, st));
}

PermuteArgs permute_args(const moe_config &c, const int32_t *ids, int T, int32_t *counts, int32_t *offsets,
                         int32_t *perm, int32_t *inv_perm, const WsLayout &L, void *ws)
{
    PermuteArgs pa{};
    pa.ids = ids;
    pa.hist = ws_at<int32_t>(ws, L.hist);
    pa.counts = counts;
    pa.offsets = offsets;
    pa.perm = perm;
    pa.inv_perm = inv_perm;
    pa.nwork = ws_at<int32_t>(ws, L.nwork);
    pa.work_dec = ws_at<WorkItem>(ws, L.work_dec);
    pa.work_g1 = ws_at<WorkItem>(ws, L.work_g1);
    pa.work_g2 = ws_at<WorkItem>(ws, L.work_g2);
    pa.status = ws_at<int>(ws, L.status);
    pa.T = T;
    pa.E = c.n_experts;
    pa.k = c.top_k;
    pa.nblk = L.nblk;
    pa.has_shared = c.has_shared;
    pa.build_work = 1;
    pa.small_tiles = prefill_small_fits(c.hidden, c.inter, qcode(c)) ? 1 : 0;
    pa.max_items[0] = L.max_wd;
    pa.max_items[1] = L.max_w1;
    pa.max_items[2] = L.max_w2;
    return pa;
}

ExpertArgs expert_args(const moe_config &c, const moe_weights &w, const uint16_t *x, int T, const uint16_t *p,
                       const uint16_t *w_s, const int32_t *offsets, const int32_t *perm, float *acc,
                       const WsLayout &L, void *ws)
{
    ExpertArgs ea{};
    ea.x = x;
    ea.gate = dev(w.gate);
    ea.up = dev(w.up);
    ea.down = dev(w.down);
    if (c.has_shared) {
        ea.s_gate = dev(w.s_gate);
        ea.s_up = dev(w.s_up);
        ea.s_down = dev(w.s_down);
    }
    ea.offsets = offsets;
    ea.perm = perm;
    ea.nwork = ws_at<int32_t>(ws, L.nwork);
    ea.h = ws_at<uint16_t>(ws, L.h);
    ea.yslot = ws_at<float>(ws, L.yslot);
    ea.xe = ws_at<int>(ws, L.xe);
    ea.p = p;
    ea.w_s = w_s;
    ea.acc = acc;
    ea.status = ws_at<int>(ws, L.status);
    ea.T = T;
    ea.H = c.hidden;
    ea.I = c.inter;
    ea.E = c.n_experts;
    ea.k = c.top_k;
    ea.has_shared = c.has_shared;
    ea.bits = qcode(c);
    return ea;
}

// The fixed-order sum of every token's slot outputs (ea.yslot; routed slot f in row pos[f], or row f
// when pos is null): into y (rounded once) or added to ea.acc.
int enqueue_slot_sum(const moe_config &c, const ExpertArgs &ea, uint16_t *y, cudaStream_t st,
                     const int32_t *pos = nullptr)
{
    ReduceArgs r{};
    r.yslot = ea.yslot;
    r.pos = pos;
    r.status = ea.status;
    r.p = ea.p;
    r.w_s = ea.w_s;
    r.acc = ea.acc;
    r.y = y;
    r.T = ea.T;
    r.H = c.hidden;
    r.k = c.top_k;
    r.has_shared = c.has_shared;
    return cuda_rc(launch_slot_sum(r, st));
}

// Decode expert kernels; the sum lands in y (rounded) or is added to acc.
int enqueue_decode_experts(const moe_config &c, ExpertArgs ea, const WsLayout &L, void *ws, uint16_t *y,
                           cudaStream_t st)
{
    ea.work = ws_at<WorkItem>(ws, L.work_dec);
    ea.max_items = L.max_wd;
    int rc = cuda_rc(launch_decode_gateup(ea, st));
    if (rc) return rc;
    rc = cuda_rc(launch_decode_down(ea, st));
    if (rc) return rc;
    return enqueue_slot_sum(c, ea, y, st);
}

// Prefill expert GEMMs.  Each slot's expert output goes to the workspace's slot buffer (rows in
// expert-sorted position order); pos (the inverse of perm: routed slot f -> position) then locates
// the slots of every token, which are summed in a fixed order into y (rounded once) or added to acc;
// or, for the stage outputs (stages), gathered in slot order into yslot_out (when non-null) with h
// to h_out, and nothing is summed.
int enqueue_prefill_experts(const moe_config &c, const ExpertArgs &ea, const WsLayout &L, void *ws, uint16_t *y,
                            const int32_t *pos, cudaStream_t st, bool stages = false, float *h_out = nullptr,
                            float *yslot_out = nullptr)
{
    PrefillArgs a{};
    a.x = ea.x;
    a.x16 = ws_at<uint16_t>(ws, L.x16);
    a.xsum = ws_at<float>(ws, L.xsum);
    a.xe = ws_at<int>(ws, L.xe);
    a.h_out = h_out;
    a.yslot = ea.yslot;
    a.hsum = ws_at<float>(ws, L.hsum);
    a.hs = ws_at<uint16_t>(ws, L.h);
    a.gate = ea.gate;
    a.up = ea.up;
    a.down = ea.down;
    a.s_gate = ea.s_gate;
    a.s_up = ea.s_up;
    a.s_down = ea.s_down;
    a.nwork = ea.nwork;
    a.offsets = ea.offsets;
    a.perm = ea.perm;
    a.work_g1 = ws_at<WorkItem>(ws, L.work_g1);
    a.work_g2 = ws_at<WorkItem>(ws, L.work_g2);
    a.status = ea.status;
    a.T = ea.T;
    a.H = c.hidden;
    a.I = c.inter;
    a.E = c.n_experts;
    a.k = c.top_k;
    a.has_shared = c.has_shared;
    a.max_w1 = L.max_w1;
    a.max_w2 = L.max_w2;
    a.bits = qcode(c);
    a.wait_limit = wait_limit_of(c);
    const int rc = cuda_rc(launch_prefill_experts(a, st));
    if (rc) return rc;
    if (stages)
        return yslot_out ? cuda_rc(launch_slot_gather(ea.yslot, pos, yslot_out, ea.T, c.hidden, c.top_k, c.has_shared,
                                                      ea.status, st))
                         : MOE_OK;
    return enqueue_slot_sum(c, ea, y, st, pos);
}

// Arguments of the fused decode kernel common to all of its callers.
FusedDecodeArgs fused_args(const moe_config &c, const moe_weights &w, const uint16_t *x, int T, const WsLayout &L,
                           void *ws)
{
    FusedDecodeArgs fa{};
    fa.x = x;
    fa.r_codes = w.router.codes;
    fa.r_scales = w.router.scales;
    fa.r_biases = w.router.biases;
    fa.v = c.has_shared ? w.shared_gate_vec : nullptr;
    fa.gate = dev(w.gate);
    fa.up = dev(w.up);
    fa.down = dev(w.down);
    if (c.has_shared) {
        fa.s_gate = dev(w.s_gate);
        fa.s_up = dev(w.s_up);
        fa.s_down = dev(w.s_down);
    }
    fa.down_packed = w.down_packed;
    fa.s_down_packed = c.has_shared ? w.s_down_packed : nullptr;
    fa.logits64 = ws_at<unsigned long long>(ws, L.logits);
    fa.p_glob = ws_at<uint16_t>(ws, L.p);
    fa.ws_glob = ws_at<uint16_t>(ws, L.w_s);
    fa.part = ws_at<float>(ws, L.dpart);
    fa.hsum = ws_at<float>(ws, L.dhsum);
    fa.sync = ws_at<int>(ws, L.status);
    fa.status = ws_at<int>(ws, L.status);
    fa.trace = ws_at<unsigned long long>(ws, L.trace);
    fa.T = T;
    fa.H = c.hidden;
    fa.I = c.inter;
    fa.E = c.n_experts;
    fa.k = c.top_k;
    fa.has_shared = c.has_shared;
    fa.wait_limit = wait_limit_of(c);
    return fa;
}

bool fused_fits(const moe_config &c, int T)
{
    return c.bits == 4 && c.format == MOE_FORMAT_AFFINE && T >= 1 && T <= kDecodeMaxTok &&
           decode_fused_fits(T, c.hidden, c.inter, c.n_experts, c.top_k, c.has_shared);
}

bool weights_ok(const moe_config &c, const moe_weights *w, bool need_router, bool need_experts)
{
    if (!w) return false;
    if (!aligned16_or_null(w->down_packed) || !aligned16_or_null(w->s_down_packed)) return false;
    if (need_router && !qmat_ok(w->router)) return false;
    if (need_experts) {
        const bool nv = c.format == MOE_FORMAT_NVFP4;
        if (!qmat_ok(w->gate, nv) || !qmat_ok(w->up, nv) || !qmat_ok(w->down, nv)) return false;
        if (c.has_shared && (!qmat_ok(w->s_gate, nv) || !qmat_ok(w->s_up, nv) || !qmat_ok(w->s_down, nv)))
            return false;
    }
    return true;
}

}  // namespace

extern "C" {

const char *moe_status_string(int status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE: return "device-side index out of range";
    default: return "unknown status";
    }
}

int moe_check_config(const moe_config *c)
{
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->hidden <= 0 || c->inter <= 0 || c->n_experts <= 0 || c->top_k <= 0) return MOE_ERR_INVALID_ARG;
    if (c->group != kGroup || (c->bits != 4 && c->bits != 8) || c->router_bits != 8) return MOE_ERR_UNSUPPORTED;
    if (c->format != MOE_FORMAT_AFFINE && !(c->format == MOE_FORMAT_NVFP4 && c->bits == 4)) return MOE_ERR_UNSUPPORTED;
    if (c->hidden % 64 || c->inter % 64 || c->hidden > 8192 || c->inter > 4096) return MOE_ERR_UNSUPPORTED;
    if (c->n_experts > kMaxExperts || c->top_k > kMaxTopK || c->top_k > c->n_experts) return MOE_ERR_UNSUPPORTED;
    if (c->has_shared != 0 && c->has_shared != 1) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int moe_workspace_size(const moe_config *cfg, int T, size_t *bytes)
{
    const int rc = check_common(cfg, T);
    if (rc) return rc;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = ws_layout(*cfg, T).total;
    return MOE_OK;
}

int moe_route(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int T, const float *router_bias,
              const float *logits_in, float *logits_out, int32_t *ids, uint16_t *p, uint16_t *w_shared, void *ws,
              size_t ws_bytes, void *stream)
{
    int rc = check_common(cfg, T);
    if (rc) return rc;
    if (!w || !aligned16(x) || !aligned16(ids) || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (!aligned16_or_null(router_bias) || !aligned16_or_null(logits_in) || !aligned16_or_null(logits_out) ||
        !aligned16_or_null(w_shared))
        return MOE_ERR_INVALID_ARG;
    if (!logits_in && !weights_ok(*cfg, w, true, false)) return MOE_ERR_INVALID_ARG;
    if (cfg->has_shared && w_shared && !aligned16(w->shared_gate_vec)) return MOE_ERR_INVALID_ARG;
    WsLayout L;
    if ((rc = check_ws(cfg, T, ws, ws_bytes, &L))) return rc;
    if (T == 0) return MOE_OK;
    auto st = static_cast<cudaStream_t>(stream);
    float *logits = logits_out ? logits_out : ws_at<float>(ws, L.logits);
    return enqueue_route(*cfg, *w, x, T, router_bias, logits_in, logits, ids, p, w_shared, L, ws, st);
}

int moe_permute(const moe_config *cfg, const int32_t *ids, int T, int32_t *counts, int32_t *offsets,
                int32_t *perm, int32_t *inv_perm, void *ws, size_t ws_bytes, void *stream)
{
    int rc = check_common(cfg, T);
    if (rc) return rc;
    if (!aligned16(ids) || !aligned16(counts) || !aligned16(offsets) || !aligned16(perm) || !aligned16(inv_perm))
        return MOE_ERR_INVALID_ARG;
    WsLayout L;
    if ((rc = check_ws(cfg, T, ws, ws_bytes, &L))) return rc;
    auto st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        rc = cuda_rc(cudaMemsetAsync(counts, 0, sizeof(int32_t) * cfg->n_experts, st));
        if (!rc) rc = cuda_rc(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (cfg->n_experts + 1), st));
        return rc;
    }
    HistArgs ha{};
    ha.ids = ids;
    ha.hist = ws_at<int32_t>(ws, L.hist);
    ha.status = ws_at<int>(ws, L.status);
    ha.T = T;
    ha.E = cfg->n_experts;
    ha.k = cfg->top_k;
    ha.nblk = L.nblk;
    if ((rc = cuda_rc(launch_hist(ha, st)))) return rc;
    return cuda_rc(launch_permute(permute_args(*cfg, ids, T, counts, offsets, perm, inv_perm, L, ws), st));
}

int moe_expert_ffn(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int T, const int32_t *ids,
                   const uint16_t *p, const uint16_t *w_shared, const int32_t *counts, const int32_t *offsets,
                   const int32_t *perm, float *acc, int path, void *ws, size_t ws_bytes, void *stream)
{
    int rc = check_common(cfg, T);
    if (rc) return rc;
    if (!weights_ok(*cfg, w, false, true) || !aligned16(x) || !aligned16(ids) || !aligned16(p) ||
        !aligned16(counts) || !aligned16(offsets) || !aligned16(perm) || !aligned16(acc))
        return MOE_ERR_INVALID_ARG;
    if (cfg->has_shared && !aligned16(w_shared)) return MOE_ERR_INVALID_ARG;
    if (path < MOE_PATH_AUTO || path > MOE_PATH_PREFILL) return MOE_ERR_INVALID_ARG;
    WsLayout L;
    if ((rc = check_ws(cfg, T, ws, ws_bytes, &L))) return rc;
    if (T == 0) return MOE_OK;
    auto st = static_cast<cudaStream_t>(stream);
    WorklistArgs wa{};
    wa.counts = counts;
    wa.nwork = ws_at<int32_t>(ws, L.nwork);
    wa.work_dec = ws_at<WorkItem>(ws, L.work_dec);
    wa.work_g1 = ws_at<WorkItem>(ws, L.work_g1);
    wa.work_g2 = ws_at<WorkItem>(ws, L.work_g2);
    wa.status = ws_at<int>(ws, L.status);
    wa.T = T;
    wa.E = cfg->n_experts;
    wa.has_shared = cfg->has_shared;
    wa.small_tiles = prefill_small_fits(cfg->hidden, cfg->inter, qcode(*cfg)) ? 1 : 0;
    wa.max_items[0] = L.max_wd;
    wa.max_items[1] = L.max_w1;
    wa.max_items[2] = L.max_w2;
    const int rp = resolve_path(*cfg, path, T);
    if (rp == MOE_PATH_DECODE && fused_fits(*cfg, T)) {
        FusedDecodeArgs fa = fused_args(*cfg, *w, x, T, L, ws);
        fa.ids_in = ids;
        fa.p_in = p;
        fa.ws_in = cfg->has_shared ? w_shared : nullptr;
        fa.acc = acc;
        return cuda_rc(launch_decode_fused(fa, st));
    }
    if ((rc = cuda_rc(launch_worklist(wa, st)))) return rc;
    ExpertArgs ea = expert_args(*cfg, *w, x, T, p, w_shared, offsets, perm, acc, L, ws);
    if (rp == MOE_PATH_DECODE) return enqueue_decode_experts(*cfg, ea, L, ws, nullptr, st);
    int32_t *pos = ws_at<int32_t>(ws, L.inv_perm);     // routed slot -> expert-sorted position
    if ((rc = cuda_rc(launch_invert_perm(perm, pos, T * cfg->top_k, ea.status, st)))) return rc;
    return enqueue_prefill_experts(*cfg, ea, L, ws, nullptr, pos, st);
}

int moe_combine(const moe_config *cfg, int T, const float *acc, uint16_t *y, void *stream)
{
    int rc = check_common(cfg, T);
    if (rc) return rc;
    if (!aligned16(acc) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    return cuda_rc(launch_combine(acc, y, (size_t)T * cfg->hidden, static_cast<cudaStream_t>(stream)));
}

int moe_forward(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int T, const float *router_bias,
                const float *logits_in, uint16_t *y, int32_t *ids_out, uint16_t *p_out, uint16_t *w_shared_out,
                int path, void *ws, size_t ws_bytes, void *stream)
{
    int rc = check_common(cfg, T);
    if (rc) return rc;
    if (!weights_ok(*cfg, w, logits_in == nullptr, true) || !aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    if (cfg->has_shared && !aligned16(w->shared_gate_vec)) return MOE_ERR_INVALID_ARG;
    if (!aligned16_or_null(router_bias) || !aligned16_or_null(logits_in) || !aligned16_or_null(ids_out) ||
        !aligned16_or_null(p_out) || !aligned16_or_null(w_shared_out))
        return MOE_ERR_INVALID_ARG;
    if (path < MOE_PATH_AUTO || path > MOE_PATH_PREFILL) return MOE_ERR_INVALID_ARG;
    WsLayout L;
    if ((rc = check_ws(cfg, T, ws, ws_bytes, &L))) return rc;
    if (T == 0) return MOE_OK;
    const int rp = resolve_path(*cfg, path, T);
    auto st = static_cast<cudaStream_t>(stream);
    if (rp == MOE_PATH_DECODE && fused_fits(*cfg, T)) {
        // the whole layer in one cooperative launch
        FusedDecodeArgs fa = fused_args(*cfg, *w, x, T, L, ws);
        fa.router_bias = logits_in ? nullptr : router_bias;
        fa.logits_in = logits_in;
        fa.ids_out = ids_out;
        fa.p_out = p_out;
        fa.ws_out = w_shared_out;
        fa.y = y;
        return cuda_rc(launch_decode_fused(fa, st));
    }
    int32_t *ids = ids_out ? ids_out : ws_at<int32_t>(ws, L.ids);
    uint16_t *p = p_out ? p_out : ws_at<uint16_t>(ws, L.p);
    uint16_t *w_s = w_shared_out ? w_shared_out : ws_at<uint16_t>(ws, L.w_s);
    float *logits = ws_at<float>(ws, L.logits);
    if ((rc = enqueue_route(*cfg, *w, x, T, router_bias, logits_in, logits_in ? nullptr : logits, ids, p, w_s, L,
                            ws, st)))
        return rc;
    int32_t *counts = ws_at<int32_t>(ws, L.counts), *offsets = ws_at<int32_t>(ws, L.offsets);
    int32_t *perm = ws_at<int32_t>(ws, L.perm), *inv_perm = ws_at<int32_t>(ws, L.inv_perm);
    if ((rc = cuda_rc(launch_permute(permute_args(*cfg, ids, T, counts, offsets, perm, inv_perm, L, ws), st))))
        return rc;
    ExpertArgs ea = expert_args(*cfg, *w, x, T, p, w_s, offsets, perm, ws_at<float>(ws, L.acc), L, ws);
    if (rp == MOE_PATH_DECODE) return enqueue_decode_experts(*cfg, ea, L, ws, y, st);
    return enqueue_prefill_experts(*cfg, ea, L, ws, y, inv_perm, st);
}

int moe_get_device_status(void *ws, size_t ws_bytes, void *stream, int *device_status)
{
    if (!aligned16(ws) || ws_bytes < kHeaderBytes || !device_status) return MOE_ERR_INVALID_ARG;
    auto st = static_cast<cudaStream_t>(stream);
    int hdr[kHeaderBytes / sizeof(int)];
    int rc = cuda_rc(cudaStreamSynchronize(st));
    if (!rc) rc = cuda_rc(cudaMemcpy(hdr, ws, kHeaderBytes, cudaMemcpyDeviceToHost));
    if (rc) return rc;
    const int v = hdr[0];
    // status word and counters to zero; the epoch moves on, so that logits a kernel published
    // under the old one can never pass for the next launch's
    const int epoch = hdr[kSyncEpoch] + 1;
    for (int &h : hdr) h = 0;
    hdr[kSyncEpoch] = epoch;
    rc = cuda_rc(cudaMemcpy(ws, hdr, kHeaderBytes, cudaMemcpyHostToDevice));
    if (rc) return rc;
    *device_status = v;
    return MOE_OK;
}

int moe_pack_down(const moe_config *cfg, const moe_weights *w, uint8_t *down_packed, uint8_t *s_down_packed,
                  void *stream)
{
    int rc = check_common(cfg, 0);
    if (rc) return rc;
    if (!w || !aligned16(w->down.codes) || !aligned16(down_packed) || !aligned16_or_null(s_down_packed))
        return MOE_ERR_INVALID_ARG;
    if (cfg->inter % kDecodeSlice || cfg->bits != 4 || cfg->format != MOE_FORMAT_AFFINE) return MOE_ERR_UNSUPPORTED;
    auto st = static_cast<cudaStream_t>(stream);
    rc = cuda_rc(launch_pack_down(w->down.codes, down_packed, cfg->n_experts, cfg->hidden, cfg->inter, st));
    if (rc || !cfg->has_shared || !s_down_packed) return rc;
    if (!aligned16(w->s_down.codes)) return MOE_ERR_INVALID_ARG;
    return cuda_rc(launch_pack_down(w->s_down.codes, s_down_packed, 1, cfg->hidden, cfg->inter, st));
}

int moe_expert_stages(const moe_config *cfg, const moe_weights *w, const uint16_t *x, int T, const int32_t *ids,
                      const int32_t *counts, const int32_t *offsets, const int32_t *perm, float *h_out,
                      float *yslot_out, int path, void *ws, size_t ws_bytes, void *stream)
{
    int rc = check_common(cfg, T);
    if (rc) return rc;
    if (!weights_ok(*cfg, w, false, true) || !aligned16(x) || !aligned16(ids) || !aligned16_or_null(h_out) ||
        !aligned16_or_null(yslot_out))
        return MOE_ERR_INVALID_ARG;
    if (path < MOE_PATH_AUTO || path > MOE_PATH_PREFILL) return MOE_ERR_INVALID_ARG;
    WsLayout L;
    if ((rc = check_ws(cfg, T, ws, ws_bytes, &L))) return rc;
    if (T == 0 || (!h_out && !yslot_out)) return MOE_OK;
    auto st = static_cast<cudaStream_t>(stream);
    const int rp = resolve_path(*cfg, path, T);
    if (rp == MOE_PATH_DECODE && fused_fits(*cfg, T)) {
        FusedDecodeArgs fa = fused_args(*cfg, *w, x, T, L, ws);
        fa.ids_in = ids;
        fa.p_in = ws_at<uint16_t>(ws, L.p);     // weights are not applied: any values serve
        fa.ws_in = nullptr;
        fa.h_out = h_out;
        fa.yslot_out = yslot_out;
        fa.stages_only = 1;
        return cuda_rc(launch_decode_fused(fa, st));
    }
    if (rp == MOE_PATH_DECODE) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(counts) || !aligned16(offsets) || !aligned16(perm)) return MOE_ERR_INVALID_ARG;
    // prefill: the grouped GEMMs of moe_expert_ffn, h per slot from the gate/up epilogue and the
    // unweighted expert output per slot from the down epilogue (no accumulator)
    WorklistArgs wa{};
    wa.counts = counts;
    wa.nwork = ws_at<int32_t>(ws, L.nwork);
    wa.work_dec = ws_at<WorkItem>(ws, L.work_dec);
    wa.work_g1 = ws_at<WorkItem>(ws, L.work_g1);
    wa.work_g2 = ws_at<WorkItem>(ws, L.work_g2);
    wa.status = ws_at<int>(ws, L.status);
    wa.T = T;
    wa.E = cfg->n_experts;
    wa.has_shared = cfg->has_shared;
    wa.small_tiles = prefill_small_fits(cfg->hidden, cfg->inter, qcode(*cfg)) ? 1 : 0;
    wa.max_items[0] = L.max_wd;
    wa.max_items[1] = L.max_w1;
    wa.max_items[2] = L.max_w2;
    if ((rc = cuda_rc(launch_worklist(wa, st)))) return rc;
    // the weights are not applied: any values serve (the workspace's own p and w_s rows)
    ExpertArgs ea = expert_args(*cfg, *w, x, T, ws_at<uint16_t>(ws, L.p), ws_at<uint16_t>(ws, L.w_s), offsets, perm,
                                ws_at<float>(ws, L.acc), L, ws);
    int32_t *pos = ws_at<int32_t>(ws, L.inv_perm);     // routed slot -> expert-sorted position
    if ((rc = cuda_rc(launch_invert_perm(perm, pos, T * cfg->top_k, ea.status, st)))) return rc;
    return enqueue_prefill_experts(*cfg, ea, L, ws, nullptr, pos, st, true, h_out, yslot_out);
}

int moe_decode_timeline(const moe_config *cfg, int T, void *ws, size_t ws_bytes, void *stream,
                        unsigned long long *host_stamps, int max_ctas, int *n_ctas)
{
    int rc = check_common(cfg, T);
    if (rc) return rc;
    if (!host_stamps || !n_ctas || max_ctas < 0) return MOE_ERR_INVALID_ARG;
    WsLayout L;
    if ((rc = check_ws(cfg, T, ws, ws_bytes, &L))) return rc;
    const int n = (int)decode_fused_trace_ctas();
    if (n <= 0 || n > kTraceMaxCtas) return MOE_ERR_CUDA;
    *n_ctas = n;
    const int m = n < max_ctas ? n : max_ctas;
    rc = cuda_rc(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    if (!rc && m > 0)
        rc = cuda_rc(cudaMemcpy(host_stamps, ws_at<unsigned long long>(ws, L.trace),
                                sizeof(unsigned long long) * kTraceStamps * (size_t)m, cudaMemcpyDeviceToHost));
    return rc;
}

}  // extern "C"
