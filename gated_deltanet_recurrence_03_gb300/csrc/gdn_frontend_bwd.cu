// The backward pass through the fused front end of the GatedDeltaNet shell ("Transformer by Hand,
// ch. 7", listing "qwen/deltanet.py", GatedDeltaNet.forward and its parts table): the l2 norm of q and
// k (GDN_NORMALIZE_QK) and the gates formed from the raw projections a, b (GDN_RAW_GATES):
//     x_n = r x,  r = (x . x + 1e-6)^(-1/2)                  dx = r dx_n - r^3 (x . dx_n) x
//     g = -exp(A_log) softplus(a + dt_bias)                   da = dg (-exp(A_log)) sigmoid(a + dt_bias)
//     beta = sigmoid(b)                                       db = dbeta beta (1 - beta)
//     dA_log = sum over tokens of dg g,  d dt_bias = sum over tokens of da   (per value head)
// The recurrence's backward differentiates the fp32 values the forward kernels form in registers, and
// a post-pass maps its gradients back to the raw inputs in place.  For bf16 inputs with dk = dv = 128
// its kernels run on the raw inputs with the front end inside (per-row l2 scalars, gates formed in
// fp32); for other shapes a pre-pass first writes the front end's outputs (normalised q, k, the gates,
// and v, dout) as fp32 into the workspace and every kernel runs in fp32 on those copies.
#include <algorithm>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr float kL2Eps = 1e-6f;
constexpr int kRowThreads = 256;   // 8 rows (one warp each) per block

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// x_n = x / sqrt(x . x + eps) per row of d values, fp32 out; one warp per row.
template <typename TT>
__global__ void __launch_bounds__(kRowThreads)
fe_l2_fwd_kernel(const TT* __restrict__ x, float* __restrict__ xn, long long rows, int d) {
    const long long row = (long long)blockIdx.x * (kRowThreads / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const TT* xr = x + row * d;
    float ss = 0.f;
    for (int i = lane; i < d; i += 32) {
        const float f = to_f32(xr[i]);
        ss = fmaf(f, f, ss);
    }
#pragma unroll
    for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float r = rsqrtf(ss + kL2Eps);
    for (int i = lane; i < d; i += 32) xn[row * d + i] = to_f32(xr[i]) * r;
}

// dx = r dx_n - r^3 (x . dx_n) x in place over dx_n, per row of d values; one warp per row.
template <typename TT>
__global__ void __launch_bounds__(kRowThreads)
fe_l2_bwd_kernel(const TT* __restrict__ x, float* __restrict__ dx, long long rows, int d) {
    const long long row = (long long)blockIdx.x * (kRowThreads / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const TT* xr = x + row * d;
    float* dr = dx + row * d;
    float ss = 0.f, xd = 0.f;
    for (int i = lane; i < d; i += 32) {
        const float f = to_f32(xr[i]);
        ss = fmaf(f, f, ss);
        xd = fmaf(f, dr[i], xd);
    }
#pragma unroll
    for (int m = 16; m; m >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, m);
        xd += __shfl_xor_sync(0xffffffffu, xd, m);
    }
    const float r = rsqrtf(ss + kL2Eps), c = r * r * r * xd;
    for (int i = lane; i < d; i += 32) dr[i] = fmaf(r, dr[i], -c * to_f32(xr[i]));
}

// fp32 copy of n values.
template <typename TT>
__global__ void fe_widen_kernel(const TT* __restrict__ x, float* __restrict__ y, long long n) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        y[i] = to_f32(x[i]);
}

// The gates per (token, value head), fp32: formed from a, b when A_log is given, else widened.
template <typename TT>
__global__ void fe_gates_fwd_kernel(const TT* __restrict__ ga, const TT* __restrict__ bb, const float* __restrict__ A_log,
                                    const float* __restrict__ dt_bias, float* __restrict__ g32, float* __restrict__ b32,
                                    long long n, int Hv) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        float g = to_f32(ga[i]), beta = to_f32(bb[i]);
        if (A_log) {
            const int h = (int)(i % Hv);
            gates_from_raw(g, beta, A_log[h], dt_bias[h], g, beta);
        }
        g32[i] = g;
        b32[i] = beta;
    }
}

// da, db in place over dg, dbeta; one block per value head, tokens in a fixed order, so the per-head
// sums dA_log = sum dg g and d dt_bias = sum da are deterministic.
constexpr int kGateThreads = 256;
template <typename TT>
__global__ void __launch_bounds__(kGateThreads)
fe_gates_bwd_kernel(const TT* __restrict__ a, const TT* __restrict__ b, const float* __restrict__ A_log,
                    const float* __restrict__ dt_bias, float* __restrict__ dg, float* __restrict__ dbeta,
                    float* __restrict__ grad_A_log, float* __restrict__ grad_dt_bias, long long tokens, int Hv) {
    __shared__ float red[2][kGateThreads];
    const int h = blockIdx.x, tid = threadIdx.x;
    const float al = A_log[h], dt = dt_bias[h], ea = __expf(al);
    float s_ag = 0.f, s_dt = 0.f;
    for (long long t = tid; t < tokens; t += kGateThreads) {
        const long long i = t * Hv + h;
        const float av = to_f32(a[i]), bv = to_f32(b[i]);
        float g, beta;
        gates_from_raw(av, bv, al, dt, g, beta);
        const float sig = 1.f / (1.f + __expf(-(av + dt)));
        const float dgi = dg[i], dai = -dgi * ea * sig;
        dg[i] = dai;
        dbeta[i] = dbeta[i] * beta * (1.f - beta);
        s_ag = fmaf(dgi, g, s_ag);
        s_dt += dai;
    }
    red[0][tid] = s_ag;
    red[1][tid] = s_dt;
    __syncthreads();
    for (int w = kGateThreads / 2; w > 0; w >>= 1) {
        if (tid < w) {
            red[0][tid] += red[0][tid + w];
            red[1][tid] += red[1][tid + w];
        }
        __syncthreads();
    }
    if (tid == 0) {
        if (grad_A_log) grad_A_log[h] = red[0][0];
        if (grad_dt_bias) grad_dt_bias[h] = red[1][0];
    }
}

// The same over all value heads at once (Hv <= 256): thread (r, h) of a block of Hv x R threads takes
// tokens b R + r, b R + r + NB R, ... of head h (coalesced rows of Hv gates), and each block writes its
// per-head sums of dg g and da, added over its R threads in a fixed order, to pa[b][h], pd[b][h];
// column_sum_kernel then adds the blocks in a fixed order.
constexpr int kGateRows = 256;
template <typename TT>
__global__ void __launch_bounds__(kGateRows)
fe_gates_bwd_rows_kernel(const TT* __restrict__ a, const TT* __restrict__ b, const float* __restrict__ A_log,
                         const float* __restrict__ dt_bias, float* __restrict__ dg, float* __restrict__ dbeta,
                         float* __restrict__ pa, float* __restrict__ pd, long long tokens, int Hv, int R) {
    __shared__ float red[2][kGateRows];
    const int tid = threadIdx.x, h = tid % Hv, r = tid / Hv;
    const long long NB = gridDim.x;
    float s_ag = 0.f, s_dt = 0.f;
    if (r < R) {
        const float al = A_log[h], dt = dt_bias[h], ea = __expf(al);
        for (long long t = (long long)blockIdx.x * R + r; t < tokens; t += NB * R) {
            const long long i = t * Hv + h;
            const float av = to_f32(a[i]), bv = to_f32(b[i]);
            float g, beta;
            gates_from_raw(av, bv, al, dt, g, beta);
            const float sig = 1.f / (1.f + __expf(-(av + dt)));
            const float dgi = dg[i], dai = -dgi * ea * sig;
            dg[i] = dai;
            dbeta[i] = dbeta[i] * beta * (1.f - beta);
            s_ag = fmaf(dgi, g, s_ag);
            s_dt += dai;
        }
    }
    red[0][tid] = s_ag;
    red[1][tid] = s_dt;
    __syncthreads();
    if (tid < Hv) {
        float x = 0.f, y = 0.f;
        for (int q = 0; q < R; ++q) {
            x += red[0][q * Hv + tid];
            y += red[1][q * Hv + tid];
        }
        pa[(size_t)blockIdx.x * Hv + tid] = x;
        pd[(size_t)blockIdx.x * Hv + tid] = y;
    }
}

unsigned grid_for(long long n, int threads) {
    const long long b = (n + threads - 1) / threads;
    return (unsigned)std::min<long long>(std::max<long long>(b, 1), 1 << 20);
}

struct FeLayout {
    size_t q, k, v, dout, g, beta, total;
};

FeLayout fe_layout(long long ttot, int Hqk, int Hv, int dk, int dv) {
    FeLayout L{};
    size_t off = 0;
    const auto take = [&](size_t& field, size_t floats) {
        field = off;
        off = round256(off + floats * sizeof(float));
    };
    take(L.q, (size_t)ttot * Hqk * dk);
    take(L.k, (size_t)ttot * Hqk * dk);
    take(L.v, (size_t)ttot * Hv * dv);
    take(L.dout, (size_t)ttot * Hv * dv);
    take(L.g, (size_t)ttot * Hv);
    take(L.beta, (size_t)ttot * Hv);
    L.total = off;
    return L;
}

template <typename TT>
cudaError_t run_frontend_backward(const BackwardArgs& in, unsigned flags, const float* A_log, const float* dt_bias,
                                  float* grad_A_log, float* grad_dt_bias, size_t core_bytes) {
    const bool packed = in.cu_seqlens != nullptr;
    const long long ttot = packed ? (long long)in.T : (long long)in.B * in.T;
    const FeLayout L = fe_layout(ttot, in.Hqk, in.Hv, in.dk, in.dv);
    uint8_t* base = static_cast<uint8_t*>(in.workspace) + round256(core_bytes);
    float* q32 = reinterpret_cast<float*>(base + L.q);
    float* k32 = reinterpret_cast<float*>(base + L.k);
    float* v32 = reinterpret_cast<float*>(base + L.v);
    float* do32 = reinterpret_cast<float*>(base + L.dout);
    float* g32 = reinterpret_cast<float*>(base + L.g);
    float* b32 = reinterpret_cast<float*>(base + L.beta);
    const bool norm = (flags & GDN_NORMALIZE_QK) != 0, raw = (flags & GDN_RAW_GATES) != 0;
    const long long qrows = ttot * in.Hqk, gates = ttot * in.Hv, vals = gates * in.dv;
    cudaStream_t s = in.stream;
    const TT* q = static_cast<const TT*>(in.q);
    const TT* k = static_cast<const TT*>(in.k);
    const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool inside = sizeof(TT) == 2 && in.dk == 128 && in.dv == 128 && al16(in.q) && al16(in.k) && al16(in.dout);
    if (ttot > 0 && !inside) {
        if (norm) {
            const unsigned blocks = (unsigned)((qrows + kRowThreads / 32 - 1) / (kRowThreads / 32));
            fe_l2_fwd_kernel<TT><<<blocks, kRowThreads, 0, s>>>(q, q32, qrows, in.dk);
            fe_l2_fwd_kernel<TT><<<blocks, kRowThreads, 0, s>>>(k, k32, qrows, in.dk);
        } else {
            fe_widen_kernel<TT><<<grid_for(qrows * in.dk, 256), 256, 0, s>>>(q, q32, qrows * in.dk);
            fe_widen_kernel<TT><<<grid_for(qrows * in.dk, 256), 256, 0, s>>>(k, k32, qrows * in.dk);
        }
        fe_widen_kernel<TT><<<grid_for(vals, 256), 256, 0, s>>>(static_cast<const TT*>(in.v), v32, vals);
        fe_widen_kernel<TT><<<grid_for(vals, 256), 256, 0, s>>>(static_cast<const TT*>(in.dout), do32, vals);
        fe_gates_fwd_kernel<TT><<<grid_for(gates, 256), 256, 0, s>>>(
            static_cast<const TT*>(in.g), static_cast<const TT*>(in.beta), raw ? A_log : nullptr, dt_bias, g32, b32,
            gates, in.Hv);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    BackwardArgs a = in;
    cudaError_t e;
    if (inside) {   // bf16 at the tensor-core shape: every kernel on the raw inputs with the front end inside
        a.flags = flags;
        a.A_log = A_log;
        a.dt_bias = dt_bias;
        e = launch_backward(a);
    } else {   // every kernel in fp32 on the copies
        a.q = q32; a.k = k32; a.v = v32; a.dout = do32; a.g = g32; a.beta = b32;
        a.dtype = GDN_F32;
        a.flags = 0;
        e = launch_backward(a);
    }
    if (e != cudaSuccess) return e;
    if (norm && ttot > 0) {
        const unsigned blocks = (unsigned)((qrows + kRowThreads / 32 - 1) / (kRowThreads / 32));
        fe_l2_bwd_kernel<TT><<<blocks, kRowThreads, 0, s>>>(q, in.grad_q, qrows, in.dk);
        fe_l2_bwd_kernel<TT><<<blocks, kRowThreads, 0, s>>>(k, in.grad_k, qrows, in.dk);
    }
    if (raw && in.Hv <= kGateRows) {   // also for no tokens: the parameter gradients are then zero
        // the per-block sums go to the gate copies' region (free once the recurrence's backward has run;
        // each of its two arrays holds ttot x Hv floats, at least NB x Hv)
        const int R = kGateRows / in.Hv;
        const long long NB = std::min<long long>((ttot + R - 1) / R, 1184);
        if (NB > 0)
            fe_gates_bwd_rows_kernel<TT><<<(unsigned)NB, in.Hv * R, 0, s>>>(
                static_cast<const TT*>(in.g), static_cast<const TT*>(in.beta), A_log, dt_bias, in.grad_g,
                in.grad_beta, g32, b32, ttot, in.Hv, R);
        const unsigned cb = (unsigned)((in.Hv + 31) / 32);
        if (grad_A_log) column_sum_kernel<<<cb, kColSumThreads, 0, s>>>(g32, NB, in.Hv, grad_A_log);
        if (grad_dt_bias) column_sum_kernel<<<cb, kColSumThreads, 0, s>>>(b32, NB, in.Hv, grad_dt_bias);
    } else if (raw) {
        fe_gates_bwd_kernel<TT><<<in.Hv, kGateThreads, 0, s>>>(
            static_cast<const TT*>(in.g), static_cast<const TT*>(in.beta), A_log, dt_bias, in.grad_g, in.grad_beta,
            grad_A_log, grad_dt_bias, ttot, in.Hv);
    }
    return cudaGetLastError();
}

}  // namespace

size_t frontend_backward_bytes(int B, int T, int Hqk, int Hv, int dk, int dv, bool packed) {
    const long long ttot = packed ? (long long)T : (long long)B * T;
    return fe_layout(ttot, Hqk, Hv, dk, dv).total;
}

cudaError_t launch_frontend_backward(const BackwardArgs& a, unsigned flags, const float* A_log, const float* dt_bias,
                                     float* grad_A_log, float* grad_dt_bias, size_t core_bytes) {
    return a.dtype == GDN_BF16
               ? run_frontend_backward<__nv_bfloat16>(a, flags, A_log, dt_bias, grad_A_log, grad_dt_bias, core_bytes)
               : run_frontend_backward<float>(a, flags, A_log, dt_bias, grad_A_log, grad_dt_bias, core_bytes);
}

}  // namespace gdn
