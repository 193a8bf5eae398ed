/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet recurrence library (libgdn.so).
 *
 * The operation (per sequence, per value head h, state S: dk x dv, fp32):
 *
 *     S_t = a_t S_{t-1} + beta_t k_t (v_t - a_t S_{t-1}^T k_t)^T,   a_t = exp(g_t)
 *     o_t = scale * S_t^T q_t
 *
 * as stated in "Transformer by Hand, ch. 7 -- Gated DeltaNet: the token-by-token
 * recurrence", section "The formula", and computed step by step (decay, look up
 * with k, write the difference times beta, read with q) by the delta_rule
 * listing of section "qwen/deltanet.py" of the same chapter.  Value head h uses
 * query/key head floor(h / (Hv / Hqk)), the repeat_interleave of the
 * GatedDeltaNet shell in the same listing.  The chunk-parallel prefill computes
 * the same result up to rounding ("mathematically equivalent to the token loop",
 * learn-llm page "linear attention", remark on flash-linear-attention).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is CALLER-OWNED DEVICE memory, contiguous, row-major.
 *   q, k, v, out and the states are 16-byte aligned; g and beta are aligned to
 *   their element size.  The library never allocates, frees or retains device
 *   memory; scratch space is passed in as opts->workspace.
 * - Calls are asynchronous on opts->stream: a return of GDN_OK means the work was
 *   validated and enqueued.  Device-side failures (a bounded wait that ran out)
 *   are read with gdn_check_device_status().
 * - Argument errors are detected on the host before anything is enqueued; nothing
 *   is written in that case.
 * - The values of g (finite, <= 0) and beta (in [0, 1]) are the caller's
 *   contract; they are not checked.  Kernels never read or write outside the
 *   buffers described by the sizes, whatever the values (cu_seqlens entries are
 *   clamped to [0, T]).
 * - Thread safety: calls on different streams may run concurrently; a workspace
 *   must not be shared by calls that overlap on the device.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, Hv % Hqk != 0 ... */
    GDN_ERR_UNSUPPORTED = 2, /* head dims or chunk outside the supported set, wrong GPU */
    GDN_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed (see gdn_last_error) */
    GDN_ERR_TIMEOUT = 4,     /* a bounded device-side wait ran out (gdn_check_device_status) */
    GDN_ERR_WORKSPACE = 5    /* workspace missing or smaller than the size query asked for */
} gdn_status_t;

typedef enum gdn_dtype {
    GDN_F32 = 0,  /* q, k, v, g, beta and out are float */
    GDN_BF16 = 1  /* q, k, v, g, beta and out are bfloat16; the state is always float */
} gdn_dtype_t;

/* opts->flags */
#define GDN_NORMALIZE_QK 0x1u /* divide q and k by sqrt(sum x^2 + 1e-6) inside the kernel
                                 (the l2norm step of delta_rule); off: inputs are used as given */
#define GDN_RAW_GATES 0x2u    /* the g and beta arguments hold the raw per-token projections a and b of
                                 the GatedDeltaNet shell ("qwen/deltanet.py", forward): the kernels form
                                 beta = sigmoid(b) and g = -exp(A_log[h]) * softplus(a + dt_bias[h]) in
                                 fp32; opts->A_log and opts->dt_bias ([Hv] float) are then required */
#define GDN_OUTPUT_GATE 0x4u  /* out = RMSNorm(o) * norm_weight * silu(z) per (token, value head), the
                                 gated normalisation of the shell (GatedRMSNorm(out, z)): o is divided by
                                 sqrt(mean over dv of o^2 + norm_eps); opts->z ([..., Hv, dv] like out,
                                 dtype) and opts->norm_weight ([dv] float) are then required */

typedef struct gdn_opts {
    int dtype;                  /* gdn_dtype_t of q, k, v, g, beta, out.  Default GDN_BF16. */
    int chunk;                  /* prefill chunk length: 16, 32 or 64 (0 -> 64; others rejected).
                                   Every chunk length gives the token loop's result up to rounding
                                   (the chunked form is the loop regrouped), and both chunked kernel
                                   families are built on 64-token tensor-core tiles: they serve all
                                   three values with 64-token chunks, so results do not depend on it. */
    float scale;                /* multiplies every output o_t.  Default 1.0f. */
    unsigned flags;             /* GDN_NORMALIZE_QK | GDN_RAW_GATES | GDN_OUTPUT_GATE, default 0 */
    const int32_t* cu_seqlens;  /* prefill only: DEVICE pointer to num_seqs+1 int32 token offsets
                                   (0 = cu[0] <= cu[1] <= ... <= cu[num_seqs] = T) of packed
                                   sequences; requires B == 1.  NULL: B sequences of T tokens. */
    int num_seqs;               /* number of packed sequences when cu_seqlens != NULL */
    void* workspace;            /* DEVICE scratch of >= gdn_chunk_fwd_workspace_size() bytes,
                                   256-byte aligned; may be NULL when that size is 0 */
    size_t workspace_bytes;
    void* stream;               /* cudaStream_t to enqueue on; NULL = legacy default stream */
    void** events;              /* optional cudaEvent_t[num_events]: events[0] is recorded before
                                   the first kernel of the call and events[i] after kernel i
                                   (kernel-level timing); NULL = none */
    int num_events;
    const float* A_log;         /* [Hv] per-head log forgetting speed (GDN_RAW_GATES), DEVICE */
    const float* dt_bias;       /* [Hv] per-head bias added to a (GDN_RAW_GATES), DEVICE */
    const void* z;              /* output gate input, same shape and dtype as out (GDN_OUTPUT_GATE), DEVICE */
    const float* norm_weight;   /* [dv] (GDN_OUTPUT_GATE), DEVICE */
    float norm_eps;             /* GDN_OUTPUT_GATE epsilon; default 1e-6 */
    float* grad_A_log;          /* gdn_recurrent_bwd with GDN_RAW_GATES: [Hv] dL/dA_log out, DEVICE; NULL = not computed */
    float* grad_dt_bias;        /* gdn_recurrent_bwd with GDN_RAW_GATES: [Hv] dL/ddt_bias out, DEVICE; NULL = not computed */
} gdn_opts_t;

/* Fill *opts with the defaults listed above. */
void gdn_opts_init(gdn_opts_t* opts);

/*
 * gdn_chunk_fwd -- chunked prefill over whole sequences.
 *
 *   q, k     [B, T, Hqk, dk]  dtype          query / key (unit length unless GDN_NORMALIZE_QK)
 *   v        [B, T, Hv, dv]   dtype
 *   g        [B, T, Hv]       dtype          log decay, a_t = exp(g_t)
 *   beta     [B, T, Hv]       dtype          write strength
 *   S0       [nseq, Hv, dk, dv] float or NULL (zero state); nseq = B, or num_seqs when packed
 *   out      [B, T, Hv, dv]   dtype          written for every token (rounded to nearest even)
 *   S_final  [nseq, Hv, dk, dv] float or NULL (not written); may equal S0 (in-place update)
 *
 * Supported: dk, dv in {32, 64, 128}; Hv a multiple of Hqk; B, T >= 0.  T = 0 copies S0 to
 * S_final (zeros when S0 is NULL).  Three kernel families, chosen in this order (opts->chunk does
 * not take part in the choice: the two chunked families block in 64-token chunks for every value):
 *   - bf16 inputs with dk = dv = 128: the tcgen05 tensor-core path; it needs the workspace
 *     (GDN_ERR_WORKSPACE if missing or too small).  Its two kernels run back to back, the second
 *     launched with programmatic stream serialisation so that its set-up overlaps the first one's
 *     last CTAs; an event in opts->events[1] (recorded between them) makes it a plain launch;
 *   - other inputs, when the workspace is at least gdn_chunk_fwd_workspace_size() bytes (256-byte
 *     aligned): the same chunk algebra on split-tf32 tensor-core MMAs in fp32 accuracy,
 *     GDN_NORMALIZE_QK and GDN_RAW_GATES included;
 *   - otherwise the token-serial CUDA-core kernel, which needs no workspace.
 * out must not overlap any input.
 *
 * Errors: GDN_ERR_INVALID_ARG for null required pointers, negative sizes, Hv % Hqk != 0,
 * pointers not 16-byte aligned, cu_seqlens with B != 1 or num_seqs < 1; GDN_ERR_UNSUPPORTED for
 * head dims or a chunk outside the sets above or a device that is not sm_103; GDN_ERR_WORKSPACE
 * when the tensor-core path is selected and the workspace is missing or too small;
 * GDN_ERR_CUDA when a launch fails.
 */
gdn_status_t gdn_chunk_fwd(const void* q, const void* k, const void* v, const void* g,
                           const void* beta, const float* S0, void* out, float* S_final, int B,
                           int T, int Hqk, int Hv, int dk, int dv, const gdn_opts_t* opts);

/* Bytes of device workspace gdn_chunk_fwd needs for these sizes and options (0 if none). */
size_t gdn_chunk_fwd_workspace_size(int B, int T, int Hqk, int Hv, int dk, int dv,
                                    const gdn_opts_t* opts);

/*
 * gdn_recurrent_step -- one decode step: one new token for each of N sequences.
 *
 *   q, k   [N, Hqk, dk] dtype;  v [N, Hv, dv] dtype;  g, beta [N, Hv] dtype
 *   S      [N, Hv, dk, dv] float, read and UPDATED IN PLACE (the state carried between calls,
 *          as delta_rule takes S in and returns the final S)
 *   out    [N, Hv, dv] dtype
 *
 * One pass over the state: each (sequence, head) table is read once and written once.
 * Supported: dk, dv in {32, 64, 128}; Hv a multiple of Hqk; N >= 0 (N = 0 is a no-op).
 * opts->chunk, cu_seqlens and workspace are ignored.  Errors as for gdn_chunk_fwd.
 */
gdn_status_t gdn_recurrent_step(const void* q, const void* k, const void* v, const void* g,
                                const void* beta, float* S, void* out, int N, int Hqk, int Hv,
                                int dk, int dv, const gdn_opts_t* opts);

/*
 * gdn_chunk_fwd_noalloc -- gdn_chunk_fwd for callers that cannot allocate device memory.
 * (No counterpart in the pages: it is a service of this library.)
 *
 * Same arguments, layouts and results as gdn_chunk_fwd; opts->workspace and workspace_bytes are
 * ignored.  The scratch the tensor-core path needs comes from a 64 MiB array built into the
 * library, which every GPU that loads the library holds until the process exits.  Meant for
 * callers that must not call cudaMalloc/cudaFree at this point (a host framework that owns all
 * device memory, a fixed memory budget, code that must not synchronise the device).  The call
 * allocates nothing.
 *
 * Limit: on the tensor-core path, problems whose gdn_chunk_fwd_workspace_size() exceeds 64 MiB
 * are rejected with GDN_ERR_WORKSPACE before anything is launched (for 32 value heads of dim 128
 * that is about 40 chunks of 64 tokens, ~2.5k tokens, per call); other shapes that large run the
 * token-serial kernel.  The 64 MiB are committed on a device when the library's module that
 * holds the array is loaded there: with CUDA's default lazy module loading that is the first call
 * of this entry point on that device (which also looks up the array's device address), with
 * CUDA_MODULE_LOADING=EAGER it is context creation.  A caller that owns nearly all device memory
 * should therefore make its first call early, before the rest of the memory goes to its pool, and
 * before any stream capture; if loading fails the call returns GDN_ERR_CUDA with CUDA's reason in
 * gdn_last_error().  On a device that is not sm_103 it returns GDN_ERR_UNSUPPORTED, as
 * gdn_chunk_fwd does.  All calls on a device share the array, which keeps the previous call's
 * contents (no part of it needs to start at zero); calls that overlap on the GPU race on it, so
 * order them.
 */
gdn_status_t gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                   const void* beta, const float* S0, void* out, float* S_final,
                                   int B, int T, int Hqk, int Hv, int dk, int dv,
                                   const gdn_opts_t* opts);

/*
 * gdn_causal_conv1d_fwd -- the short causal convolution that feeds q, k and v: depthwise (each
 * channel on its own), window K, then SiLU, as in the GatedDeltaNet shell of "Transformer by Hand,
 * ch. 7" (conv1d with groups = channels and padding K - 1, cut to the first T outputs, SiLU):
 *     y[t, c] = silu( sum_{i<K} w[c, i] * x[t - (K - 1) + i, c] )
 * Inputs before a sequence's first token come from cache_in (zeros when NULL).
 *
 *   x          [B, T, C] dtype, token rows x_stride elements apart (0 = C; a channel slice of a wider
 *              packed projection can be passed directly), 16-byte aligned
 *   w          [C, K] float; w[c, K-1] weighs the current token
 *   cache_in   [nseq, K-1, C] dtype or NULL: the K-1 inputs preceding each sequence, oldest first
 *   y          [B, T, C] dtype; must not overlap x or either cache
 *   cache_out  [nseq, K-1, C] dtype or NULL: the last K-1 inputs of each sequence (what a decode step
 *              needs next; for sequences shorter than K-1 the older entries come from cache_in)
 * nseq = B, or num_seqs with opts->cu_seqlens (B == 1, packed sequences, state reset at each start).
 * Supported: C a multiple of 8, 1 <= K <= 4.  opts->dtype, cu_seqlens, num_seqs, stream are used.
 */
gdn_status_t gdn_causal_conv1d_fwd(const void* x, long long x_stride, const float* w, const void* cache_in,
                                   void* y, void* cache_out, int B, int T, int C, int K,
                                   const gdn_opts_t* opts);

/*
 * gdn_causal_conv1d_step -- one decode token per sequence through the same convolution, with the
 * 3-token (K-1) cache the learn-llm page describes ("at inference the most recent 3 tokens' inputs
 * are cached"):  x [N, C] (rows x_stride apart), cache [N, K-1, C] read and updated in place (shifted
 * by one token), y [N, C].
 */
gdn_status_t gdn_causal_conv1d_step(const void* x, long long x_stride, const float* w, void* cache, void* y,
                                    int N, int C, int K, const gdn_opts_t* opts);

/*
 * gdn_causal_conv1d_fwd_qkv / gdn_causal_conv1d_step_qkv -- the same convolutions over the packed
 * projection of the GatedDeltaNet shell (its q, k and v channels side by side in one row: q in
 * [0, Cq), k in [Cq, Cq + Ck), v in [Cq + Ck, C), C = Cq + Ck + Cv), in one launch, writing the three
 * channel ranges to three dense tensors -- the layouts gdn_chunk_fwd and gdn_recurrent_step take:
 *
 *   x          [B, T, C] (fwd) or [N, C] (step) dtype, rows x_stride elements apart (0 = C)
 *   w          [C, K] float, the channels in the same q | k | v order
 *   y_q, y_k, y_v  [B, T, Cq], [B, T, Ck], [B, T, Cv] (fwd) or [N, Cq], [N, Ck], [N, Cv] (step) dtype
 *   caches     as for the single-output calls, over all C channels
 * Cq, Ck, Cv positive multiples of 8; the results are bit-identical to the single-output call
 * followed by a split of y.  Errors and options as for the single-output calls.
 */
gdn_status_t gdn_causal_conv1d_fwd_qkv(const void* x, long long x_stride, const float* w, const void* cache_in,
                                       void* y_q, void* y_k, void* y_v, void* cache_out, int B, int T, int Cq,
                                       int Ck, int Cv, int K, const gdn_opts_t* opts);
gdn_status_t gdn_causal_conv1d_step_qkv(const void* x, long long x_stride, const float* w, void* cache, void* y_q,
                                        void* y_k, void* y_v, int N, int Cq, int Ck, int Cv, int K,
                                        const gdn_opts_t* opts);

/*
 * gdn_causal_conv1d_bwd -- gradients through gdn_causal_conv1d_fwd, given grad_y = dL/dy and, for a
 * decode that continues from the outgoing cache, grad_cache_out = dL/dcache_out.  With xp a sequence's
 * inputs padded on the left by its K-1 cached inputs, u_t = sum_i w[c, i] xp[t + i] and
 * du_t = grad_y[t] silu'(u_t):
 *     grad_x (and grad_cache_in for the cached rows) = sum_i w[c, i] du_{p - i} at input position p,
 *     plus grad_cache_out for the inputs the outgoing cache holds;
 *     grad_w[c, i] = sum over all tokens of du_t xp[t + i].
 *   x, x_stride, w, cache_in, B, T, C, K, cu_seqlens / num_seqs, dtype: as gdn_causal_conv1d_fwd
 *   grad_y           [B, T, C] dtype, dense (the gradients of the q, k and v slices side by side for
 *                    the packed projection), 16-byte aligned
 *   grad_cache_out   [nseq, K-1, C] dtype or NULL (no loss on the outgoing cache)
 *   grad_x           [B, T, C] float, dense, 16-byte aligned (overwritten)
 *   grad_w           [C, K] float or NULL (not computed); summed over 64-token slots in a fixed order
 *                    through opts->workspace (256-byte aligned, gdn_causal_conv1d_bwd_workspace_size
 *                    bytes; GDN_ERR_WORKSPACE if missing)
 *   grad_cache_in    [nseq, K-1, C] float or NULL (not written), 16-byte aligned
 * Deterministic.  Asynchronous on opts->stream; events[0] / [1] around the kernels.
 */
size_t gdn_causal_conv1d_bwd_workspace_size(int B, int T, int C, int K, const gdn_opts_t* opts);
gdn_status_t gdn_causal_conv1d_bwd(const void* x, long long x_stride, const float* w, const void* cache_in,
                                   const void* grad_y, const void* grad_cache_out, float* grad_x, float* grad_w,
                                   float* grad_cache_in, int B, int T, int C, int K, const gdn_opts_t* opts);

/*
 * gdn_recurrent_bwd -- the backward pass: gradients of a loss L(out, S_final) of gdn_chunk_fwd with
 * respect to q, k, v, g, beta and S0, given grad_out = dL/dout and grad_S_final = dL/dS_final.  It is
 * the adjoint of the token loop of "Transformer by Hand, ch. 7" (section "The formula"), which the
 * learn-llm "linear attention" page trains through autograd:
 *     lam = dL/dS_t;  lam += scale q_t do_t^T;  dq_t = scale S_t do_t;  dk_t = lam u_t + S_{t-1} dp;
 *     dv_t = beta_t du;  dbeta_t = du.(v_t - a_t p_t);  dg_t = a_t (<lam, S_{t-1}> - beta_t du.p_t);
 *     lam <- a_t lam + k_t dp^T;  dS0 = lam at the start,
 * with p_t = S_{t-1}^T k_t, u_t = beta_t (v_t - a_t p_t), du = lam^T k_t, dp = -a_t beta_t du.
 *
 *   q, k, v, g, beta, S0, B, T, Hqk, Hv, dk, dv, cu_seqlens/num_seqs, scale, dtype: as gdn_chunk_fwd
 *   grad_out       [B, T, Hv, dv] in the inputs' dtype
 *   grad_S_final   [nseq, Hv, dk, dv] float, or NULL (no loss on the final state)
 *   grad_q, grad_k [B, T, Hqk, dk] float (a query/key head sums over the value heads that read it)
 *   grad_v         [B, T, Hv, dv] float;  grad_g, grad_beta [B, T, Hv] float
 *   grad_S0        [nseq, Hv, dk, dv] float, or NULL (not written)
 * Gradients are always fp32.  Pointers need only element alignment.
 * opts->flags may hold GDN_NORMALIZE_QK and GDN_RAW_GATES (GDN_OUTPUT_GATE: GDN_ERR_UNSUPPORTED): the
 * gradients are then those of the forward with the same flags, with respect to its raw inputs -- the
 * unnormalised q, k (dx = r dx_n - r^3 (x . dx_n) x, r = (x . x + 1e-6)^-1/2) and the raw projections
 * a, b passed as g, beta (da = dg (-exp(A_log)) sigmoid(a + dt_bias), db = dbeta beta (1 - beta)) --
 * and, when opts->grad_A_log / grad_dt_bias are not NULL, [Hv] fp32 sums over all tokens of dg g and
 * of da (overwritten, deterministic order).  With either flag the inputs' front-end outputs are formed
 * in fp32: for bf16 inputs with dk = dv = 128 (16-byte aligned q, k, grad_out) inside the kernels,
 * which read the raw inputs and form the per-row l2 scalars and the gates in fp32; otherwise as fp32
 * copies in the workspace (gdn_recurrent_bwd_workspace_size grows accordingly), on which the whole
 * backward runs in fp32 (the split-tf32 kernels).  It is computed through the chunked form
 * of the loop (64-token chunks): the workspace (256-byte aligned, gdn_recurrent_bwd_workspace_size
 * bytes) holds per (chunk, value head) the chunk's UT inverse, decay-masked Q K^T, W, U, decay
 * prefix sums, the state at the chunk start and its adjoint, and dU, all fp32; GDN_ERR_WORKSPACE if
 * missing or too small.  For bf16 inputs with dk = dv = 128 and 16-byte aligned q, k and grad_out the
 * two chunk chains run on the tcgen05 tensor cores (fp32 accuracy through three-part bf16 operand
 * splits).  Asynchronous on opts->stream; events[0] before the four kernels and events[i] after
 * kernel i (1: WY factors, 2: forward chain, 3: adjoint chain, 4: chunk-local gradients).
 */
size_t gdn_recurrent_bwd_workspace_size(int B, int T, int Hqk, int Hv, int dk, int dv, const gdn_opts_t* opts);
gdn_status_t gdn_recurrent_bwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                               const float* S0, const void* grad_out, const float* grad_S_final, float* grad_q,
                               float* grad_k, float* grad_v, float* grad_g, float* grad_beta, float* grad_S0,
                               int B, int T, int Hqk, int Hv, int dk, int dv, const gdn_opts_t* opts);

/*
 * gdn_output_gate_fwd -- the output gate of the GatedDeltaNet shell on its own ("Transformer by Hand,
 * ch. 7", listing "qwen/deltanet.py": out = GatedRMSNorm(o, z); its parts table: normalised per head,
 * then times silu(z)), per row of dv values (one token and value head):
 *     y_j = o_j / sqrt(mean_j(o_j^2) + eps) * norm_weight_j * silu(z_j)
 * the same pass gdn_chunk_fwd applies with GDN_OUTPUT_GATE, for callers that keep the recurrence's
 * output o (a training step needs it for the backward below).
 *   o, z, y        [rows, dv] dtype (opts->dtype), 16-byte aligned; y may equal o (in place)
 *   norm_weight    [dv] float;  eps = opts->norm_eps
 * Supported dv: 32, 64, 128.  Asynchronous on opts->stream; events[0] / [1] around the kernel.
 */
gdn_status_t gdn_output_gate_fwd(const void* o, const void* z, const float* norm_weight, void* y, long long rows,
                                 int dv, const gdn_opts_t* opts);

/*
 * gdn_output_gate_bwd -- gradients through gdn_output_gate_fwd given grad_y = dL/dy: with
 * inv = (mean(o^2) + eps)^-1/2, o_hat = o inv and gy = grad_y norm_weight silu(z), per row
 *     grad_o = inv (gy - o_hat mean(gy o_hat)),   grad_z = grad_y o_hat norm_weight silu'(z),
 * and grad_norm_weight = sum over all rows of grad_y o_hat silu(z).
 *   o, z, grad_y            [rows, dv] dtype, 16-byte aligned
 *   grad_o, grad_z          [rows, dv] float (overwritten), 16-byte aligned
 *   grad_norm_weight        [dv] float (overwritten), or NULL (not computed); its sum over rows is
 *                           taken in a fixed order through opts->workspace (256-byte aligned,
 *                           gdn_output_gate_bwd_workspace_size bytes; GDN_ERR_WORKSPACE if missing)
 * Deterministic.  Asynchronous on opts->stream; events[0] / [1] around the kernels.
 */
size_t gdn_output_gate_bwd_workspace_size(long long rows, int dv, const gdn_opts_t* opts);
gdn_status_t gdn_output_gate_bwd(const void* o, const void* z, const float* norm_weight, const void* grad_y,
                                 float* grad_o, float* grad_z, float* grad_norm_weight, long long rows, int dv,
                                 const gdn_opts_t* opts);

/* Synchronise `stream` (cudaStream_t, NULL = legacy), then read and clear the device status word
 * that kernels set when a bounded wait runs out.  GDN_OK if clear, GDN_ERR_TIMEOUT if set,
 * GDN_ERR_CUDA if the synchronisation itself failed. */
gdn_status_t gdn_check_device_status(void* stream);

/* Static description of a status code. */
const char* gdn_status_string(gdn_status_t status);

/* Message of the last failure on the calling thread ("" if none). */
const char* gdn_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
