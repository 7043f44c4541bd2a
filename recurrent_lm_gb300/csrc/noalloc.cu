// la_prefix_prefill_noalloc: the JRT-RNN prefix prefill for callers that
// cannot allocate device memory at call time.
//
// la_prefix_prefill needs scratch memory for the per-segment partial prefix
// states, which its caller passes in.  Some callers have no way to provide it:
// code that runs where an allocation is not allowed or would stall (a
// latency-critical serving loop that must not trigger the implicit
// synchronisation of cudaMalloc, or a plug-in whose host process hands all
// device memory to its own allocator and exposes none to plug-ins).  For them
// this file holds a fixed scratch buffer in device memory, reserved when the
// library's module is loaded on a device and kept until the process exits.
//
// The entry point itself allocates nothing: it looks up the device address of
// the buffer (once per device) and runs the ordinary prefix prefill with it.
#include <mutex>

#include "la_internal.h"

namespace {

// Largest la_prefix_workspace_size() this entry point accepts.
constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

// Only device code may use this name directly; host code must use the address
// returned by cudaGetSymbolAddress (the host-side symbol is a stand-in, not a
// device pointer).
static __device__ __align__(256) unsigned char g_la_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch buffer on the current device (looked up on
// the first call made with that device current).
la_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_la_noalloc_scratch) != cudaSuccess || p == nullptr) return LA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return LA_OK;
}

}  // namespace

extern "C" {

size_t la_noalloc_scratch_bytes(void) { return kScratchBytes; }

la_status la_prefix_prefill_noalloc(const void *q, const void *k, const void *v, const void *k_e,
                                    const void *v_e, int64_t M, const float *s0, const float *z0,
                                    void *y, float *s_out, float *z_out, int64_t B, int64_t H,
                                    int64_t N, int d_feat, int d_v, la_dtype dtype, float eps,
                                    la_stream_t stream) {
    // the full workspace when it fits, else the prefix partial states alone
    // (the prefill then runs without split heads)
    const size_t need = la::prefix_workspace_min(B, H, M);
    if (need > kScratchBytes) return LA_ERR_SCRATCH_TOO_SMALL;
    void *scratch = nullptr;
    if (need > 0) {
        la_status st = scratch_address(&scratch);
        if (st != LA_OK) return st;
    }
    return la_prefix_prefill(q, k, v, k_e, v_e, M, s0, z0, y, s_out, z_out, scratch,
                             need > 0 ? kScratchBytes : 0, B, H, N, d_feat, d_v, dtype, eps, stream);
}

}  // extern "C"
