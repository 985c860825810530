// moe_forward_decode_static: the decode layer for callers that cannot allocate.
//
// Some callers of this library cannot call cudaMalloc: code that runs inside
// another engine's enqueue callback, where that engine owns every byte of
// device memory, or a process that must not allocate once it has started
// (a real-time loop, a deployment that fixes its memory footprint up front).
// For them this entry point runs the same decode kernels as moe_forward, but
// its scratch is a fixed array in the library's own device memory instead of
// a caller workspace.
//
// The array is declared below at file scope.  Every GPU that loads the library
// holds it until the process exits.  Host code cannot use the array's name as a
// device address (it is a host-side stand-in), so the device address is looked
// up once per device with cudaGetSymbolAddress, on the first call made with
// that device current; make that first call before any stream capture.
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr size_t kStaticScratchBytes = 24u << 20;   // 24 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_moe_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the static scratch on the current device (looked up once).
int static_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_moe_static_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" MOE_API int moe_forward_decode_static(const moe_config *cfg, const moe_weights *w, const uint16_t *x,
                                                 int T, const float *router_bias, const float *logits_in,
                                                 uint16_t *y, int32_t *ids_out, uint16_t *p_out,
                                                 uint16_t *w_shared_out, void *stream)
{
    if (!cfg) return MOE_ERR_INVALID_ARG;
    int rc = moe_check_config(cfg);
    if (rc != MOE_OK) return rc;
    if (T < 0 || T > qmoe::kDecodeMaxTok) return MOE_ERR_INVALID_ARG;   // decode sizes only: 0 <= T <= 16
    size_t need = 0;
    if ((rc = moe_workspace_size(cfg, T, &need)) != MOE_OK) return rc;
    if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;            // layer too large for the fixed array
    void *scratch = nullptr;
    if ((rc = static_scratch(&scratch)) != MOE_OK) return rc;
    return moe_forward(cfg, w, x, T, router_bias, logits_in, y, ids_out, p_out, w_shared_out, MOE_PATH_DECODE,
                       scratch, kStaticScratchBytes, stream);
}
