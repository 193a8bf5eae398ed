// gdn_chunk_fwd_noalloc: the chunked prefill for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where they run the
// prefill: code that runs inside another framework's memory pool with a fixed budget, code
// that must not synchronise the device (cudaMalloc and cudaFree can), embedded or
// safety-certified runtimes that forbid allocation after start-up, and plugins whose host
// process owns all device memory.  The tensor-core prefill needs scratch space between its two
// kernels; this entry point takes that scratch from a fixed array compiled into the library
// instead of from the caller.
//
// The array lives in device memory of every GPU that loads the library, for the life of the
// process.  It is committed when this translation unit's module is loaded on a device: with CUDA's
// default lazy module loading that happens inside the first call of this entry point on that
// device (the cudaGetSymbolAddress below loads it), with CUDA_MODULE_LOADING=EAGER when the
// process creates its context.  A caller that owns nearly all device memory should make that first
// call early (before handing the rest of the memory to its pool) and before any stream capture.
// Its size caps the problem size; larger problems are rejected with
// GDN_ERR_WORKSPACE before anything is launched.  Every call on a device uses the same array and
// it keeps whatever the previous call wrote.  Nothing in it has to start at zero: each call
// writes every scratch byte it later reads.  Two calls whose work overlaps on the GPU (for
// example on two streams of one device) would use the array at the same time and race; order
// them on one stream or with events.
#include <cstdio>
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];

// The device address of the array on the current device.  In host code the symbol's name is
// only a host-side stand-in: its device address must be asked for, once per device, with that
// device current.
cudaError_t scratch_on_current_device(void** ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status_t gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                              const void* beta, const float* S0, void* out, float* S_final,
                                              int B, int T, int Hqk, int Hv, int dk, int dv,
                                              const gdn_opts_t* opts) {
    gdn_opts_t o;
    gdn_opts_init(&o);
    if (opts) o = *opts;
    o.workspace = nullptr;
    o.workspace_bytes = 0;
    const size_t need = gdn_chunk_fwd_workspace_size(B, T, Hqk, Hv, dk, dv, &o);
    if (need > gdn::kNoAllocScratchBytes) {
        // the chunked path of shapes off the tensor-core tile falls back to the token-serial kernel,
        // which needs no scratch; the tensor-core path has no such fallback
        if (!gdn::tc_prefill_eligible(o.dtype, dk, dv, Hqk, Hv, o.chunk, o.flags))
            return gdn_chunk_fwd(q, k, v, g, beta, S0, out, S_final, B, T, Hqk, Hv, dk, dv, &o);
        gdn::set_error_message("gdn_chunk_fwd_noalloc: this problem needs more scratch than the built-in "
                               "64 MiB array; use gdn_chunk_fwd with a caller workspace");
        return GDN_ERR_WORKSPACE;
    }
    if (need > 0) {
        // the same status as gdn_chunk_fwd on a device this library does not run on, before the
        // symbol lookup (which would fail there with a less useful CUDA error)
        const gdn_status_t dst = gdn::check_current_device();
        if (dst != GDN_OK) return dst;
        void* p = nullptr;
        const cudaError_t e = gdn::scratch_on_current_device(&p);
        if (e != cudaSuccess) {
            char msg[200];
            snprintf(msg, sizeof(msg),
                     "gdn_chunk_fwd_noalloc: cudaGetSymbolAddress of the scratch array failed "
                     "(loading the module commits the 64 MiB array): %s", cudaGetErrorString(e));
            gdn::set_error_message(msg);
            return GDN_ERR_CUDA;
        }
        o.workspace = p;
        o.workspace_bytes = gdn::kNoAllocScratchBytes;
    }
    return gdn_chunk_fwd(q, k, v, g, beta, S0, out, S_final, B, T, Hqk, Hv, dk, dv, &o);
}
