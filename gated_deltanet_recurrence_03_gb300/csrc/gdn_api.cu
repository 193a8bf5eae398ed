// C ABI of libgdn (declared in include/gdn.h): argument validation, kernel selection, device
// status word, error reporting.  Every check that can fail does so on the host before anything is
// enqueued.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "gdn_internal.cuh"

#define GDN_VERSION_MAJOR 0
#define GDN_VERSION_MINOR 3
#define GDN_VERSION_PATCH 0

namespace gdn {
namespace {

// Device status word: kernels OR kStatusTimeout into it when a bounded wait runs out.
__device__ unsigned g_status_word;

thread_local char t_last_error[256] = "";

gdn_status_t fail(gdn_status_t s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
gdn_status_t fail(gdn_status_t s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return s;
}

gdn_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int g_dev_checked[kMaxDevices];    // 0 unknown, 1 sm_103, -1 other
unsigned* g_dev_status[kMaxDevices];

// Current device must be sm_103; fetch its status word address (per device, once).
gdn_status_t device_ready(unsigned** status) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_dev_checked[dev] == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major == 10 && minor == 3) {
            void* p = nullptr;  // the symbol's device address (the host-side name is only a stand-in)
            e = cudaGetSymbolAddress(&p, g_status_word);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
            g_dev_status[dev] = static_cast<unsigned*>(p);
            g_dev_checked[dev] = 1;
        } else {
            g_dev_checked[dev] = -1;
        }
    }
    if (g_dev_checked[dev] != 1)
        return fail(GDN_ERR_UNSUPPORTED, "libgdn is built for sm_103a; device %d is not sm_103", dev);
    *status = g_dev_status[dev];
    return GDN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void* p, unsigned bytes) { return (reinterpret_cast<uintptr_t>(p) % bytes) == 0; }
unsigned elem_bytes(int dtype) { return dtype == GDN_BF16 ? 2u : 4u; }
bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

gdn_opts_t resolve(const gdn_opts_t* o) {
    gdn_opts_t r;
    gdn_opts_init(&r);
    if (o) r = *o;
    if (r.chunk == 0) r.chunk = 64;
    return r;
}

gdn_status_t check_common(int Hqk, int Hv, int dk, int dv, const gdn_opts_t& o) {
    if (Hqk <= 0 || Hv <= 0) return fail(GDN_ERR_INVALID_ARG, "head counts must be positive (Hqk=%d Hv=%d)", Hqk, Hv);
    if (Hv % Hqk != 0) return fail(GDN_ERR_INVALID_ARG, "Hv (%d) must be a multiple of Hqk (%d)", Hv, Hqk);
    if (dk <= 0 || dv <= 0) return fail(GDN_ERR_INVALID_ARG, "head dims must be positive");
    if (o.dtype != GDN_F32 && o.dtype != GDN_BF16) return fail(GDN_ERR_INVALID_ARG, "unknown dtype %d", o.dtype);
    if (o.flags & ~(GDN_NORMALIZE_QK | GDN_RAW_GATES | GDN_OUTPUT_GATE))
        return fail(GDN_ERR_INVALID_ARG, "unknown flags 0x%x", o.flags);
    if ((o.flags & GDN_OUTPUT_GATE) && (!o.z || !o.norm_weight || !aligned16(o.z) || !aligned_to(o.norm_weight, 4)))
        return fail(GDN_ERR_INVALID_ARG, "GDN_OUTPUT_GATE needs a 16-byte aligned z and an aligned norm_weight");
    if ((o.flags & GDN_OUTPUT_GATE) && !(o.norm_eps >= 0.f)) return fail(GDN_ERR_INVALID_ARG, "norm_eps must be >= 0");
    if ((o.flags & GDN_RAW_GATES) && (!o.A_log || !o.dt_bias || !aligned_to(o.A_log, 4) || !aligned_to(o.dt_bias, 4)))
        return fail(GDN_ERR_INVALID_ARG, "GDN_RAW_GATES needs aligned A_log and dt_bias");
    if (o.num_events < 0 || (o.num_events > 0 && !o.events)) return fail(GDN_ERR_INVALID_ARG, "bad event list");
    if (!dim_ok(dk) || !dim_ok(dv)) return fail(GDN_ERR_UNSUPPORTED, "head dims dk=%d dv=%d not in {32,64,128}", dk, dv);
    return GDN_OK;
}

void record(const gdn_opts_t& o, int i, cudaStream_t s) {
    if (o.events && i < o.num_events && o.events[i]) cudaEventRecord(static_cast<cudaEvent_t>(o.events[i]), s);
}

}  // namespace

void set_error_message(const char* msg) { snprintf(t_last_error, sizeof(t_last_error), "%s", msg); }

gdn_status_t check_current_device() {
    unsigned* status = nullptr;
    return device_ready(&status);
}

}  // namespace gdn

using namespace gdn;

extern "C" {

void gdn_opts_init(gdn_opts_t* o) {
    if (!o) return;
    std::memset(o, 0, sizeof(*o));
    o->dtype = GDN_BF16;
    o->chunk = 64;
    o->scale = 1.0f;
    o->norm_eps = 1e-6f;
}

int gdn_version(void) { return GDN_VERSION_MAJOR * 10000 + GDN_VERSION_MINOR * 100 + GDN_VERSION_PATCH; }

const char* gdn_last_error(void) { return t_last_error; }

const char* gdn_status_string(gdn_status_t s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported configuration";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_TIMEOUT: return "device-side wait timed out";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

}  // extern "C"

namespace {
// The chunked prefill covers every head-dim pair in {32, 64, 128}^2 with the full front end (l2 norm
// of q and k as per-row scalars, gates from raw projections); the output gate is a separate pass after
// either prefill.
bool chunked_prefill_eligible(int dk, int dv) {
    return (dk == 32 || dk == 64 || dk == 128) && (dv == 32 || dv == 64 || dv == 128);
}
}  // namespace

extern "C" {

size_t gdn_chunk_fwd_workspace_size(int B, int T, int Hqk, int Hv, int dk, int dv, const gdn_opts_t* opts) {
    const gdn_opts_t o = resolve(opts);
    if (B < 0 || T < 0 || Hqk <= 0 || Hv <= 0 || Hv % Hqk) return 0;
    const bool packed = o.cu_seqlens != nullptr;
    const int nseq = packed ? o.num_seqs : B;
    if (nseq <= 0 || T == 0) return 0;
    if (tc_prefill_eligible(o.dtype, dk, dv, Hqk, Hv, o.chunk, o.flags))
        return tc_prefill_workspace_bytes(B, T, Hv, nseq, packed);
    if (chunked_prefill_eligible(dk, dv)) return chunked_prefill_workspace_bytes(B, T, Hv, dk, dv, nseq, packed);
    return 0;
}

gdn_status_t gdn_chunk_fwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                           const float* S0, void* out, float* S_final, int B, int T, int Hqk, int Hv, int dk,
                           int dv, const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_opts_t o = resolve(opts);
    if (B < 0 || T < 0) return fail(GDN_ERR_INVALID_ARG, "B=%d T=%d must be >= 0", B, T);
    gdn_status_t st = check_common(Hqk, Hv, dk, dv, o);
    if (st != GDN_OK) return st;
    if (o.chunk != 16 && o.chunk != 32 && o.chunk != 64)
        return fail(GDN_ERR_UNSUPPORTED, "chunk %d not in {16,32,64}", o.chunk);
    const bool packed = o.cu_seqlens != nullptr;
    if (packed && (B != 1 || o.num_seqs < 1))
        return fail(GDN_ERR_INVALID_ARG, "cu_seqlens needs B == 1 and num_seqs >= 1 (B=%d num_seqs=%d)", B, o.num_seqs);
    const int nseq = packed ? o.num_seqs : B;
    const bool have_tokens = (long long)B * T > 0;
    if (have_tokens && (!q || !k || !v || !g || !beta || !out))
        return fail(GDN_ERR_INVALID_ARG, "null input/output pointer");
    const void* ptrs[] = {q, k, v, S0, out, S_final, o.cu_seqlens, o.workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(GDN_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
    if ((g && !aligned_to(g, elem_bytes(o.dtype))) || (beta && !aligned_to(beta, elem_bytes(o.dtype))))
        return fail(GDN_ERR_INVALID_ARG, "g/beta not aligned to their element size");
    if (nseq == 0) return GDN_OK;

    unsigned* status = nullptr;
    st = device_ready(&status);
    if (st != GDN_OK) return st;
    cudaStream_t stream = static_cast<cudaStream_t>(o.stream);
    const size_t state_bytes = (size_t)nseq * Hv * dk * dv * sizeof(float);

    if (!have_tokens) {  // no tokens: the final state is the initial state
        record(o, 0, stream);
        if (S_final && S_final != S0) {
            cudaError_t e = S0 ? cudaMemcpyAsync(S_final, S0, state_bytes, cudaMemcpyDeviceToDevice, stream)
                               : cudaMemsetAsync(S_final, 0, state_bytes, stream);
            if (e != cudaSuccess) return cuda_fail(e, "state copy");
        }
        record(o, 1, stream);
        return GDN_OK;
    }

    PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.S0 = S0; a.out = out; a.S_final = S_final;
    a.B = B; a.T = T; a.Hqk = Hqk; a.Hv = Hv; a.dk = dk; a.dv = dv;
    a.dtype = o.dtype; a.chunk = o.chunk; a.scale = o.scale; a.flags = o.flags;
    a.cu_seqlens = o.cu_seqlens; a.num_seqs = nseq;
    a.workspace = o.workspace; a.workspace_bytes = o.workspace_bytes;
    a.stream = stream; a.status = status;
    a.A_log = o.A_log; a.dt_bias = o.dt_bias;
    a.z = o.z; a.norm_weight = o.norm_weight; a.norm_eps = o.norm_eps;

    cudaError_t e;
    if (tc_prefill_eligible(o.dtype, dk, dv, Hqk, Hv, o.chunk, o.flags)) {
        const size_t need = tc_prefill_workspace_bytes(B, T, Hv, nseq, packed);
        if (!o.workspace || o.workspace_bytes < need)
            return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                        o.workspace ? o.workspace_bytes : (size_t)0);
        if ((reinterpret_cast<uintptr_t>(o.workspace) & 255u) != 0)
            return fail(GDN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
        e = launch_tc_prefill(a, o.events, o.num_events);
        if (e == cudaSuccess && (o.flags & GDN_OUTPUT_GATE)) {
            e = launch_output_gate(out, o.z, o.norm_weight, o.norm_eps, (long long)B * T * Hv, dv, o.dtype, stream);
            record(o, 3, stream);
        }
    } else if (chunked_prefill_eligible(dk, dv) && o.workspace &&
               (reinterpret_cast<uintptr_t>(o.workspace) & 255u) == 0 &&
               o.workspace_bytes >= chunked_prefill_workspace_bytes(B, T, Hv, dk, dv, nseq, packed)) {
        // chunked form on the split-tf32 tensor-core kernels (fp32 accuracy)
        record(o, 0, stream);
        e = launch_chunked_prefill(a);
        record(o, 1, stream);
        if (e == cudaSuccess && (o.flags & GDN_OUTPUT_GATE)) {
            e = launch_output_gate(out, o.z, o.norm_weight, o.norm_eps, (long long)B * T * Hv, dv, o.dtype, stream);
            record(o, 2, stream);
        }
    } else {   // no (or too small a) workspace: the token-serial kernel
        record(o, 0, stream);
        e = launch_recurrent_prefill(a);
        record(o, 1, stream);
        if (e == cudaSuccess && (o.flags & GDN_OUTPUT_GATE)) {
            e = launch_output_gate(out, o.z, o.norm_weight, o.norm_eps, (long long)B * T * Hv, dv, o.dtype, stream);
            record(o, 2, stream);
        }
    }
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return GDN_OK;
}

gdn_status_t gdn_recurrent_step(const void* q, const void* k, const void* v, const void* g, const void* beta,
                                float* S, void* out, int N, int Hqk, int Hv, int dk, int dv,
                                const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_opts_t o = resolve(opts);
    if (N < 0) return fail(GDN_ERR_INVALID_ARG, "N=%d must be >= 0", N);
    gdn_status_t st = check_common(Hqk, Hv, dk, dv, o);
    if (st != GDN_OK) return st;
    if (N == 0) return GDN_OK;
    if (!q || !k || !v || !g || !beta || !S || !out) return fail(GDN_ERR_INVALID_ARG, "null pointer");
    const void* ptrs[] = {q, k, v, S, out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(GDN_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
    if (!aligned_to(g, elem_bytes(o.dtype)) || !aligned_to(beta, elem_bytes(o.dtype)))
        return fail(GDN_ERR_INVALID_ARG, "g/beta not aligned to their element size");
    unsigned* status = nullptr;
    st = device_ready(&status);
    if (st != GDN_OK) return st;
    DecodeArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.S = S; a.out = out;
    a.N = N; a.Hqk = Hqk; a.Hv = Hv; a.dk = dk; a.dv = dv;
    a.dtype = o.dtype; a.scale = o.scale; a.flags = o.flags;
    a.stream = static_cast<cudaStream_t>(o.stream);
    a.A_log = o.A_log; a.dt_bias = o.dt_bias;
    a.z = o.z; a.norm_weight = o.norm_weight; a.norm_eps = o.norm_eps;
    record(o, 0, a.stream);
    cudaError_t e = launch_decode(a);
    record(o, 1, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return GDN_OK;
}

static gdn_status_t conv_common(const void* x, long long* x_stride, const float* w, int C, int K,
                                const gdn_opts_t& o) {
    if (C <= 0 || C % 8 != 0) return fail(GDN_ERR_INVALID_ARG, "C=%d must be a positive multiple of 8", C);
    if (K < 1 || K > 4) return fail(GDN_ERR_UNSUPPORTED, "kernel width K=%d not in 1..4", K);
    if (o.dtype != GDN_F32 && o.dtype != GDN_BF16) return fail(GDN_ERR_INVALID_ARG, "unknown dtype %d", o.dtype);
    if (*x_stride == 0) *x_stride = C;
    const int per16 = o.dtype == GDN_BF16 ? 8 : 4;   // elements in 16 bytes: rows must stay 16-byte aligned
    if (*x_stride < C || *x_stride % per16 != 0)
        return fail(GDN_ERR_INVALID_ARG, "x_stride=%lld must be >= C and a multiple of %d", *x_stride, per16);
    if (!x || !w) return fail(GDN_ERR_INVALID_ARG, "null x or w");
    if (!aligned16(x) || !aligned_to(w, 4)) return fail(GDN_ERR_INVALID_ARG, "x must be 16-byte aligned, w 4-byte aligned");
    return GDN_OK;
}

}  // extern "C"

namespace {

// Shared by the single-output and the q | k | v split entry points: y_k == nullptr means one output.
gdn_status_t conv_fwd_impl(const void* x, long long x_stride, const float* w, const void* cache_in, void* y,
                           void* y_k, void* y_v, int c1, int c2, void* cache_out, int B, int T, int C, int K,
                           const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_opts_t o = resolve(opts);
    if (B < 0 || T < 0) return fail(GDN_ERR_INVALID_ARG, "B=%d T=%d must be >= 0", B, T);
    const bool packed = o.cu_seqlens != nullptr;
    if (packed && (B != 1 || o.num_seqs < 1))
        return fail(GDN_ERR_INVALID_ARG, "cu_seqlens needs B == 1 and num_seqs >= 1");
    const int nseq = packed ? o.num_seqs : B;
    if (nseq == 0) return GDN_OK;
    gdn_status_t st = conv_common(x, &x_stride, w, C, K, o);
    if (st != GDN_OK) return st;
    const bool have_tokens = (long long)B * T > 0;
    if (have_tokens && (!y || (y_k && !y_v))) return fail(GDN_ERR_INVALID_ARG, "null y");
    const void* ptrs[] = {y, y_k, y_v, cache_in, cache_out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(GDN_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
    if (packed && !aligned_to(o.cu_seqlens, 4)) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
    unsigned* status = nullptr;
    st = device_ready(&status);
    if (st != GDN_OK) return st;
    ConvArgs a{};
    a.x = x; a.x_stride = x_stride; a.w = w; a.cache_in = cache_in; a.y = y; a.cache_out = cache_out;
    a.y_k = y_k; a.y_v = y_v; a.c1 = c1; a.c2 = c2;
    a.B = B; a.T = T; a.C = C; a.K = K; a.dtype = o.dtype; a.cu_seqlens = o.cu_seqlens; a.num_seqs = nseq;
    a.packed = packed; a.stream = static_cast<cudaStream_t>(o.stream); a.status = status;
    record(o, 0, a.stream);
    const cudaError_t e = launch_conv_fwd(a);
    record(o, 1, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "conv launch");
    return GDN_OK;
}

gdn_status_t conv_step_impl(const void* x, long long x_stride, const float* w, void* cache, void* y, void* y_k,
                            void* y_v, int c1, int c2, int N, int C, int K, const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_opts_t o = resolve(opts);
    if (N < 0) return fail(GDN_ERR_INVALID_ARG, "N=%d must be >= 0", N);
    if (N == 0) return GDN_OK;
    gdn_status_t st = conv_common(x, &x_stride, w, C, K, o);
    if (st != GDN_OK) return st;
    if (!y || (y_k && !y_v) || (K > 1 && !cache)) return fail(GDN_ERR_INVALID_ARG, "null y or cache");
    const void* ptrs[] = {y, y_k, y_v, cache};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(GDN_ERR_INVALID_ARG, "y and cache must be 16-byte aligned");
    unsigned* status = nullptr;
    st = device_ready(&status);
    if (st != GDN_OK) return st;
    ConvArgs a{};
    a.x = x; a.x_stride = x_stride; a.w = w; a.y = y; a.cache_out = cache;
    a.y_k = y_k; a.y_v = y_v; a.c1 = c1; a.c2 = c2;
    a.B = N; a.C = C; a.K = K; a.dtype = o.dtype; a.stream = static_cast<cudaStream_t>(o.stream);
    record(o, 0, a.stream);
    const cudaError_t e = launch_conv_step(a);
    record(o, 1, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "conv step launch");
    return GDN_OK;
}

gdn_status_t qkv_widths(int Cq, int Ck, int Cv) {
    if (Cq <= 0 || Ck <= 0 || Cv <= 0 || Cq % 8 || Ck % 8 || Cv % 8)
        return fail(GDN_ERR_INVALID_ARG, "q/k/v widths %d/%d/%d must be positive multiples of 8", Cq, Ck, Cv);
    if ((long long)Cq + Ck + Cv > INT32_MAX) return fail(GDN_ERR_INVALID_ARG, "too many channels");
    return GDN_OK;
}

}  // namespace

extern "C" {

gdn_status_t gdn_causal_conv1d_fwd(const void* x, long long x_stride, const float* w, const void* cache_in, void* y,
                                   void* cache_out, int B, int T, int C, int K, const gdn_opts_t* opts) {
    return conv_fwd_impl(x, x_stride, w, cache_in, y, nullptr, nullptr, 0, 0, cache_out, B, T, C, K, opts);
}

gdn_status_t gdn_causal_conv1d_fwd_qkv(const void* x, long long x_stride, const float* w, const void* cache_in,
                                       void* y_q, void* y_k, void* y_v, void* cache_out, int B, int T, int Cq,
                                       int Ck, int Cv, int K, const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_status_t st = qkv_widths(Cq, Ck, Cv);
    if (st != GDN_OK) return st;
    if ((long long)B * T > 0 && (!y_q || !y_k || !y_v)) return fail(GDN_ERR_INVALID_ARG, "null y_q, y_k or y_v");
    return conv_fwd_impl(x, x_stride, w, cache_in, y_q, y_k, y_v, Cq, Cq + Ck, cache_out, B, T, Cq + Ck + Cv, K,
                         opts);
}

gdn_status_t gdn_causal_conv1d_step(const void* x, long long x_stride, const float* w, void* cache, void* y, int N,
                                    int C, int K, const gdn_opts_t* opts) {
    return conv_step_impl(x, x_stride, w, cache, y, nullptr, nullptr, 0, 0, N, C, K, opts);
}

gdn_status_t gdn_causal_conv1d_step_qkv(const void* x, long long x_stride, const float* w, void* cache, void* y_q,
                                        void* y_k, void* y_v, int N, int Cq, int Ck, int Cv, int K,
                                        const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_status_t st = qkv_widths(Cq, Ck, Cv);
    if (st != GDN_OK) return st;
    if (N > 0 && (!y_q || !y_k || !y_v)) return fail(GDN_ERR_INVALID_ARG, "null y_q, y_k or y_v");
    return conv_step_impl(x, x_stride, w, cache, y_q, y_k, y_v, Cq, Cq + Ck, N, Cq + Ck + Cv, K, opts);
}

size_t gdn_causal_conv1d_bwd_workspace_size(int B, int T, int C, int K, const gdn_opts_t* opts) {
    const gdn_opts_t o = resolve(opts);
    if (B < 0 || T < 0 || C <= 0 || C % 8 || K < 1 || K > 4) return 0;
    const bool packed = o.cu_seqlens != nullptr;
    const int nseq = packed ? o.num_seqs : B;
    if (nseq <= 0) return 0;
    return conv_bwd_workspace_bytes(B, T, C, K, nseq, packed);
}

gdn_status_t gdn_causal_conv1d_bwd(const void* x, long long x_stride, const float* w, const void* cache_in,
                                   const void* grad_y, const void* grad_cache_out, float* grad_x, float* grad_w,
                                   float* grad_cache_in, int B, int T, int C, int K, const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_opts_t o = resolve(opts);
    if (B < 0 || T < 0) return fail(GDN_ERR_INVALID_ARG, "B=%d T=%d must be >= 0", B, T);
    const bool packed = o.cu_seqlens != nullptr;
    if (packed && (B != 1 || o.num_seqs < 1))
        return fail(GDN_ERR_INVALID_ARG, "cu_seqlens needs B == 1 and num_seqs >= 1");
    const int nseq = packed ? o.num_seqs : B;
    if (nseq == 0) return GDN_OK;
    gdn_status_t st = conv_common(x, &x_stride, w, C, K, o);
    if (st != GDN_OK) return st;
    const bool have_tokens = (long long)B * T > 0;
    if (have_tokens && (!grad_y || !grad_x)) return fail(GDN_ERR_INVALID_ARG, "null grad_y or grad_x");
    const void* ptrs[] = {cache_in, grad_y, grad_cache_out, grad_x, grad_cache_in};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(GDN_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
    if (grad_w && !aligned_to(grad_w, 4)) return fail(GDN_ERR_INVALID_ARG, "grad_w must be 4-byte aligned");
    if (packed && !aligned_to(o.cu_seqlens, 4)) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
    const size_t need = conv_bwd_workspace_bytes(B, T, C, K, nseq, packed);
    if (grad_w && (!o.workspace || o.workspace_bytes < need))
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    o.workspace ? o.workspace_bytes : (size_t)0);
    if (o.workspace && (reinterpret_cast<uintptr_t>(o.workspace) & 255u) != 0)
        return fail(GDN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    unsigned* status = nullptr;
    st = device_ready(&status);
    if (st != GDN_OK) return st;
    ConvArgs a{};
    a.x = x; a.x_stride = x_stride; a.w = w; a.cache_in = cache_in;
    a.B = B; a.T = T; a.C = C; a.K = K; a.dtype = o.dtype; a.cu_seqlens = o.cu_seqlens; a.num_seqs = nseq;
    a.packed = packed; a.stream = static_cast<cudaStream_t>(o.stream); a.status = status;
    record(o, 0, a.stream);
    const cudaError_t e = launch_conv_bwd(a, grad_y, grad_cache_out, grad_x, grad_w, grad_cache_in,
                                          grad_w ? o.workspace : nullptr);
    record(o, 1, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "conv backward launch");
    return GDN_OK;
}

size_t gdn_recurrent_bwd_workspace_size(int B, int T, int Hqk, int Hv, int dk, int dv, const gdn_opts_t* opts) {
    const gdn_opts_t o = resolve(opts);
    if (B < 0 || T < 0 || Hqk <= 0 || Hv <= 0 || Hv % Hqk || !dim_ok(dk) || !dim_ok(dv)) return 0;
    const bool packed = o.cu_seqlens != nullptr;
    const int nseq = packed ? o.num_seqs : B;
    if (nseq <= 0) return 0;
    const bool front_end = (o.flags & (GDN_NORMALIZE_QK | GDN_RAW_GATES)) != 0;
    size_t bytes = backward_layout(B, T, Hv, dk, dv, nseq, packed, true, front_end).total;
    if (front_end)
        bytes = ((bytes + 255) & ~(size_t)255) + frontend_backward_bytes(B, T, Hqk, Hv, dk, dv, packed);
    return bytes;
}

gdn_status_t gdn_recurrent_bwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                               const float* S0, const void* grad_out, const float* grad_S_final, float* grad_q,
                               float* grad_k, float* grad_v, float* grad_g, float* grad_beta, float* grad_S0, int B,
                               int T, int Hqk, int Hv, int dk, int dv, const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_opts_t o = resolve(opts);
    if (B < 0 || T < 0) return fail(GDN_ERR_INVALID_ARG, "B=%d T=%d must be >= 0", B, T);
    gdn_status_t st = check_common(Hqk, Hv, dk, dv, o);
    if (st != GDN_OK) return st;
    if (o.flags & ~(GDN_NORMALIZE_QK | GDN_RAW_GATES))
        return fail(GDN_ERR_UNSUPPORTED, "the backward pass has no output gate (flags 0x%x given)", o.flags);
    if ((o.flags & GDN_RAW_GATES) && (!o.A_log || !o.dt_bias))
        return fail(GDN_ERR_INVALID_ARG, "GDN_RAW_GATES needs opts->A_log and opts->dt_bias");
    const bool front_end = (o.flags & (GDN_NORMALIZE_QK | GDN_RAW_GATES)) != 0;
    const bool packed = o.cu_seqlens != nullptr;
    if (packed && (B != 1 || o.num_seqs < 1))
        return fail(GDN_ERR_INVALID_ARG, "cu_seqlens needs B == 1 and num_seqs >= 1 (B=%d num_seqs=%d)", B, o.num_seqs);
    const int nseq = packed ? o.num_seqs : B;
    const bool have_tokens = (long long)B * T > 0;
    if (have_tokens && (!q || !k || !v || !g || !beta || !grad_out || !grad_q || !grad_k || !grad_v || !grad_g ||
                        !grad_beta))
        return fail(GDN_ERR_INVALID_ARG, "null input or gradient pointer");
    const unsigned e = elem_bytes(o.dtype);
    const void* in_ptrs[] = {q, k, v, g, beta, grad_out};
    for (const void* p : in_ptrs)
        if (p && !aligned_to(p, e)) return fail(GDN_ERR_INVALID_ARG, "input %p not aligned to its element size", p);
    const void* f_ptrs[] = {S0, grad_S_final, grad_q, grad_k, grad_v, grad_g, grad_beta, grad_S0, o.cu_seqlens,
                            o.A_log, o.dt_bias, o.grad_A_log, o.grad_dt_bias};
    for (const void* p : f_ptrs)
        if (p && !aligned_to(p, 4)) return fail(GDN_ERR_INVALID_ARG, "pointer %p not 4-byte aligned", p);
    if (nseq == 0) return GDN_OK;
    const size_t core = backward_layout(B, T, Hv, dk, dv, nseq, packed, true, front_end).total;
    const size_t need =
        front_end ? ((core + 255) & ~(size_t)255) + frontend_backward_bytes(B, T, Hqk, Hv, dk, dv, packed) : core;
    if (!o.workspace || o.workspace_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    o.workspace ? o.workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(o.workspace) & 255u) != 0)
        return fail(GDN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    unsigned* status = nullptr;
    st = device_ready(&status);
    if (st != GDN_OK) return st;
    BackwardArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.S0 = S0; a.dout = grad_out; a.dS_final = grad_S_final;
    a.grad_q = grad_q; a.grad_k = grad_k; a.grad_v = grad_v; a.grad_g = grad_g; a.grad_beta = grad_beta;
    a.grad_S0 = grad_S0;
    a.B = B; a.T = T; a.Hqk = Hqk; a.Hv = Hv; a.dk = dk; a.dv = dv; a.dtype = o.dtype; a.scale = o.scale;
    a.cu_seqlens = o.cu_seqlens; a.num_seqs = nseq; a.workspace = o.workspace;
    a.stream = static_cast<cudaStream_t>(o.stream);
    a.status = status;
    a.events = o.events;
    a.num_events = o.num_events;
    record(o, 0, a.stream);
    // records events[1..4] after the four kernels of the recurrence's backward
    const cudaError_t err = front_end ? launch_frontend_backward(a, o.flags, o.A_log, o.dt_bias, o.grad_A_log,
                                                                 o.grad_dt_bias, core)
                                      : launch_backward(a);
    if (err != cudaSuccess) return cuda_fail(err, "backward launch");
    return GDN_OK;
}

namespace {
gdn_status_t gate_common(const gdn_opts_t& o, long long rows, int dv, const float* norm_weight) {
    if (rows < 0) return fail(GDN_ERR_INVALID_ARG, "rows=%lld must be >= 0", rows);
    if (dv != 32 && dv != 64 && dv != 128) return fail(GDN_ERR_UNSUPPORTED, "dv=%d: supported 32, 64, 128", dv);
    if (o.dtype != GDN_F32 && o.dtype != GDN_BF16) return fail(GDN_ERR_INVALID_ARG, "unknown dtype %d", o.dtype);
    if (!(o.norm_eps >= 0.f)) return fail(GDN_ERR_INVALID_ARG, "norm_eps must be >= 0");
    if (rows > 0 && !norm_weight) return fail(GDN_ERR_INVALID_ARG, "null norm_weight");
    return GDN_OK;
}
}  // namespace

gdn_status_t gdn_output_gate_fwd(const void* o, const void* z, const float* norm_weight, void* y, long long rows, int dv,
                                 const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_opts_t op = resolve(opts);
    gdn_status_t st = gate_common(op, rows, dv, norm_weight);
    if (st != GDN_OK) return st;
    if (rows == 0) return GDN_OK;
    if (!o || !z || !y) return fail(GDN_ERR_INVALID_ARG, "null o, z or y");
    const void* vec16[] = {o, z, y};
    for (const void* p : vec16)
        if (!aligned_to(p, 16)) return fail(GDN_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    if (!aligned_to(norm_weight, 4)) return fail(GDN_ERR_INVALID_ARG, "norm_weight not 4-byte aligned");
    unsigned* status = nullptr;
    if ((st = device_ready(&status)) != GDN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(op.stream);
    record(op, 0, s);
    const cudaError_t e = launch_output_gate_to(o, y, z, norm_weight, op.norm_eps, rows, dv, op.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "output gate launch");
    record(op, 1, s);
    return GDN_OK;
}

size_t gdn_output_gate_bwd_workspace_size(long long rows, int dv, const gdn_opts_t* opts) {
    (void)opts;
    if (rows < 0 || (dv != 32 && dv != 64 && dv != 128)) return 0;
    return output_gate_bwd_workspace_bytes(rows, dv);
}

gdn_status_t gdn_output_gate_bwd(const void* o, const void* z, const float* norm_weight, const void* grad_y,
                                 float* grad_o, float* grad_z, float* grad_norm_weight, long long rows, int dv,
                                 const gdn_opts_t* opts) {
    t_last_error[0] = 0;
    const gdn_opts_t op = resolve(opts);
    gdn_status_t st = gate_common(op, rows, dv, norm_weight);
    if (st != GDN_OK) return st;
    if (rows > 0 && (!o || !z || !grad_y || !grad_o || !grad_z))
        return fail(GDN_ERR_INVALID_ARG, "null o, z, grad_y, grad_o or grad_z");
    const void* vec16[] = {o, z, grad_y, grad_o, grad_z};
    for (const void* p : vec16)
        if (p && !aligned_to(p, 16)) return fail(GDN_ERR_INVALID_ARG, "pointer %p not 16-byte aligned", p);
    const void* f4[] = {norm_weight, grad_norm_weight};
    for (const void* p : f4)
        if (p && !aligned_to(p, 4)) return fail(GDN_ERR_INVALID_ARG, "pointer %p not 4-byte aligned", p);
    if (rows == 0 && !grad_norm_weight) return GDN_OK;
    const size_t need = output_gate_bwd_workspace_bytes(rows, dv);
    if (grad_norm_weight && rows > 0 && (!op.workspace || op.workspace_bytes < need))
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    op.workspace ? op.workspace_bytes : (size_t)0);
    if (op.workspace && (reinterpret_cast<uintptr_t>(op.workspace) & 255u) != 0)
        return fail(GDN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    unsigned* status = nullptr;
    if ((st = device_ready(&status)) != GDN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(op.stream);
    record(op, 0, s);
    const cudaError_t e = launch_output_gate_bwd(o, z, norm_weight, op.norm_eps, grad_y, grad_o, grad_z,
                                                 grad_norm_weight, op.workspace, rows, dv, op.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "output gate backward launch");
    record(op, 1, s);
    return GDN_OK;
}

gdn_status_t gdn_check_device_status(void* stream) {
    t_last_error[0] = 0;
    unsigned* status = nullptr;
    gdn_status_t st = device_ready(&status);
    if (st != GDN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, status, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (host & kStatusTimeout) return fail(GDN_ERR_TIMEOUT, "a device-side wait ran out of time");
    return GDN_OK;
}

}  // extern "C"
