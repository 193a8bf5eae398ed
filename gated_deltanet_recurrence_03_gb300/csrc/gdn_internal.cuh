// Internal interfaces of libgdn: argument bundles handed from the C ABI layer (gdn_api.cu) to the
// kernel launchers of the other translation units, and small device helpers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Device status word bits (set by kernels whose bounded waits ran out).
enum : unsigned { kStatusTimeout = 1u };

// Bounded spin: every device-side wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* g;
    const void* beta;
    const float* S0;
    void* out;
    float* S_final;
    int B, T, Hqk, Hv, dk, dv;
    int dtype;
    int chunk;
    float scale;
    unsigned flags;
    const int32_t* cu_seqlens;  // device, or nullptr
    int num_seqs;               // sequences (B, or num_seqs when packed)
    void* workspace;
    size_t workspace_bytes;
    cudaStream_t stream;
    unsigned* status;           // device status word
    const float* A_log;         // GDN_RAW_GATES
    const float* dt_bias;
    const void* z;              // GDN_OUTPUT_GATE
    const float* norm_weight;
    float norm_eps;
};

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* g;
    const void* beta;
    float* S;
    void* out;
    int N, Hqk, Hv, dk, dv;
    int dtype;
    float scale;
    unsigned flags;
    cudaStream_t stream;
    const float* A_log;         // GDN_RAW_GATES
    const float* dt_bias;
    const void* z;              // GDN_OUTPUT_GATE
    const float* norm_weight;
    float norm_eps;
};

struct ConvArgs {
    const void* x;
    long long x_stride;         // elements between consecutive token rows of x
    const float* w;             // [C, K]
    const void* cache_in;       // fwd: [nseq, K-1, C] or nullptr
    void* y;
    void* cache_out;            // fwd: [nseq, K-1, C] or nullptr; step: the cache, updated in place
    int B, T, C, K;             // step: B = number of sequences, T unused
    int dtype;
    const int32_t* cu_seqlens;
    int num_seqs;
    bool packed;
    cudaStream_t stream;
    unsigned* status;           // device status word (bounded waits)
    // Split output (the packed q | k | v projection): channels [c1, c2) go to y_k, [c2, C) to y_v, each
    // a contiguous [rows, width] tensor; y holds [0, c1).  y_k == nullptr: all C channels go to y.
    void* y_k;
    void* y_v;
    int c1, c2;
};

// Launchers (return the launch error, cudaSuccess if enqueued).
struct BackwardArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* g;
    const void* beta;
    const float* S0;            // or nullptr (zero state)
    const void* dout;           // gradient of out, v's dtype
    const float* dS_final;      // gradient of S_final, or nullptr
    float* grad_q;
    float* grad_k;
    float* grad_v;
    float* grad_g;
    float* grad_beta;
    float* grad_S0;             // or nullptr
    int B, T, Hqk, Hv, dk, dv;
    int dtype;
    float scale;
    const int32_t* cu_seqlens;
    int num_seqs;
    void* workspace;
    cudaStream_t stream;
    unsigned* status;           // device status word (bounded waits)
    void** events;              // optional: events[i] recorded after kernel i (1..4)
    int num_events;
    // The fused front end (GDN_NORMALIZE_QK, GDN_RAW_GATES; 0 = none): g and beta then hold the raw a, b.
    // Only for bf16 inputs with dk = dv = 128: every kernel then runs on the raw inputs with the front
    // end inside (per-row l2 scalars, which the WY kernel forms and keeps per chunk, and the gates formed
    // in fp32).
    unsigned flags;
    const float* A_log;
    const float* dt_bias;
};

// Workspace of the backward pass: per (chunk slot, value head) fp32 arrays T, P (C x C), W (C x dk),
// U (C x dv), G (C), chunk-start state S and its adjoint dS (dk x dv), dU (C x dv); byte offsets,
// 256-byte aligned.  `slots` = ceil(tokens / C) + sequences.
struct BwdLayout {
    long long slots;
    size_t T_off, P_off, W_off, U_off, G_off, S_off, dS_off, dU_off, R_off, total;
};
// with_r: also the per-row l2 scalars (R) of the front end, next to the adjoint arrays.
BwdLayout backward_layout(int B, int T, int Hv, int dk, int dv, int nseq, bool packed, bool adjoint,
                          bool with_r = false);
cudaError_t launch_backward(const BackwardArgs& a);
// The backward through the fused front end (GDN_NORMALIZE_QK, GDN_RAW_GATES): fp32 copies of the front
// end's outputs after the first core_bytes of a.workspace (frontend_backward_bytes more), the backward
// on them, then the gradients mapped back to the raw q, k, a, b in place; dA_log and d dt_bias into
// grad_A_log / grad_dt_bias when not NULL.
size_t frontend_backward_bytes(int B, int T, int Hqk, int Hv, int dk, int dv, bool packed);
cudaError_t launch_frontend_backward(const BackwardArgs& a, unsigned flags, const float* A_log, const float* dt_bias,
                                     float* grad_A_log, float* grad_dt_bias, size_t core_bytes);
// The backward's forward chunk chain on the tcgen05 tensor cores, for bf16 k with dk = dv = 128: the
// chunk-start states into ws_S, U = U~ - W S over ws_U (U~ read from there), the last state into
// S_final (or not).  cudaErrorNotSupported when k is not 16-byte aligned (the caller then runs the
// general chain).
cudaError_t launch_bwd_state_fwd_tc(const void* k, const float* S0, float* S_final, const float* ws_W, float* ws_U,
                                    const float* ws_G, float* ws_S, const float* ws_R, int T, int Hqk, int Hv,
                                    const int32_t* cu, int nseq, bool normalize, cudaStream_t stream,
                                    unsigned* status);
// The backward's adjoint chunk chain on the tcgen05 tensor cores (bf16 inputs, dk = dv = 128): dU and
// the chunk-end adjoints into the workspace, the gradient of S0 (or not).  cudaErrorNotSupported when
// q, k or dout is not 16-byte aligned.
cudaError_t launch_bwd_state_adj_tc(const void* q, const void* k, const void* dout, const float* dS_final,
                                    float* grad_S0, const float* ws_W, const float* ws_P, const float* ws_G,
                                    float* ws_dS, float* ws_dU, int T, int Hqk, int Hv, const int32_t* cu, int nseq,
                                    float scale, cudaStream_t stream, unsigned* status, const float* ws_R = nullptr,
                                    bool normalize = false);
// Chunked prefill for shapes outside the tensor-core path (fp32 inputs, head dims 32 / 64, front end
// included): the backward's WY kernel and forward chain plus an output kernel.
size_t chunked_prefill_workspace_bytes(int B, int T, int Hv, int dk, int dv, int nseq, bool packed);
cudaError_t launch_chunked_prefill(const PrefillArgs& a);

// The CUDA driver's cuTensorMapEncodeTiled (looked up once), or nullptr when the CUDA driver lacks it.
void* tensor_map_encoder();

cudaError_t launch_conv_fwd(const ConvArgs& a);
cudaError_t launch_conv_step(const ConvArgs& a);
// Backward of the conv + SiLU: dx [B*T, C] and dcache [nseq, K-1, C] fp32 (dcache may be NULL), dw [C, K]
// fp32 summed over 64-token slots in a fixed order through `workspace` (conv_bwd_workspace_bytes; may be
// NULL when dw is NULL).  dy is dense [B*T, C], dco (the outgoing cache's gradient) [nseq, K-1, C] or NULL,
// both in a.dtype.
size_t conv_bwd_workspace_bytes(int B, int T, int C, int K, int nseq, bool packed);
cudaError_t launch_conv_bwd(const ConvArgs& a, const void* dy, const void* dco, float* dx, float* dw, float* dcache,
                            void* workspace);
cudaError_t launch_decode(const DecodeArgs& a);
cudaError_t launch_recurrent_prefill(const PrefillArgs& a);
// out <- RMSNorm(out) * norm_weight * silu(z) over each of `rows` rows of dv values, in place.
cudaError_t launch_output_gate(void* out, const void* z, const float* w, float eps, long long rows, int dv,
                               int dtype, cudaStream_t stream);
// y <- RMSNorm(o) * norm_weight * silu(z) (in may equal out), and its backward: d_o, d_z (fp32, rows x dv)
// and, when d_w is not NULL, d_w [dv] summed over the rows in a fixed order through `workspace`
// (output_gate_bwd_workspace_bytes, 16-byte aligned).
cudaError_t launch_output_gate_to(const void* in, void* out, const void* z, const float* w, float eps, long long rows,
                                  int dv, int dtype, cudaStream_t stream);
size_t output_gate_bwd_workspace_bytes(long long rows, int dv);
cudaError_t launch_output_gate_bwd(const void* o, const void* z, const float* w, float eps, const void* dy, float* d_o,
                                   float* d_z, float* d_w, void* workspace, long long rows, int dv, int dtype,
                                   cudaStream_t stream);

// Tensor-core chunked prefill: whether it takes these arguments, its workspace, and its launch.
bool tc_prefill_eligible(int dtype, int dk, int dv, int Hqk, int Hv, int chunk, unsigned flags);
size_t tc_prefill_workspace_bytes(int B, int T, int Hv, int num_seqs, bool packed);
cudaError_t launch_tc_prefill(const PrefillArgs& a, void** events, int num_events);

// out[c] = sum over r < rows of in[r * cols + c], for c < cols, in a fixed order (deterministic): each block
// takes 32 columns; its 32 x 32 threads sum every 32nd row (warp-coalesced) and a shared-memory tree adds
// the 32 partial sums.  Launch: grid ceil(cols / 32), block kColSumThreads.
constexpr int kColSumThreads = 1024;
__global__ void column_sum_kernel(const float* __restrict__ in, long long rows, int cols, float* __restrict__ out);

// Set the calling thread's gdn_last_error() message.
void set_error_message(const char* msg);
// GDN_OK when the current device is an sm_103 GPU this library runs on; otherwise the status (and
// gdn_last_error() message) every entry point returns for it.
gdn_status_t check_current_device();

// ---------------------------------------------------------------- device helpers
template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Gates of the GatedDeltaNet shell ("Transformer by Hand, ch. 7", listing "qwen/deltanet.py",
// GatedDeltaNet.forward): beta = sigmoid(b), g = -exp(A_log) * softplus(a + dt_bias), with
// softplus(x) = max(x, 0) + log(1 + exp(-|x|)).
__device__ __forceinline__ void gates_from_raw(float a, float b, float A_log, float dt_bias, float& g, float& beta) {
    const float x = a + dt_bias;
    const float sp = fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x)));
    g = -__expf(A_log) * sp;
    beta = 1.f / (1.f + __expf(-b));
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + __expf(-z)); }

// SiLU for a result stored as bf16: z/2 (1 + tanh(z/2)) with the hardware tanh, one special-function
// op instead of two plus a division; its relative error (~2^-11 on tanh) is below bf16's 2^-9.
__device__ __forceinline__ float silu_bf16out(float z) {
    const float h = 0.5f * z;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}
template <typename T>
__device__ __forceinline__ float silu_for(float z) { return silu_f(z); }
template <>
__device__ __forceinline__ float silu_for<__nv_bfloat16>(float z) { return silu_bf16out(z); }

// Sequence i's token range [t0, t1) in the flattened token index.
__device__ __forceinline__ void seq_range(const int32_t* cu, int i, int T, long long& t0, long long& t1) {
    if (cu) {
        int a = cu[i], b = cu[i + 1];
        a = a < 0 ? 0 : (a > T ? T : a);
        b = b < a ? a : (b > T ? T : b);
        t0 = a;
        t1 = b;
    } else {
        t0 = (long long)i * T;
        t1 = t0 + T;
    }
}

}  // namespace gdn
