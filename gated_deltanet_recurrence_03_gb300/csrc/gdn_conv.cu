// Depthwise causal short convolution + SiLU ("Transformer by Hand, ch. 7", listing
// "qwen/deltanet.py": conv1d(groups = channels, kernel K, padding K - 1) cut to the first T outputs,
// then SiLU; the parts table: "each channel first sees its own previous 3 tokens"; the learn-llm page:
// at inference the layer caches the most recent 3 tokens' inputs):
//     y[t, c] = silu( sum_{i=0}^{K-1} w[c, i] * x[t - (K - 1) + i, c] )
// with x before a sequence's first token taken from that sequence's cache (or zero).
//
// Memory bound.  Each thread owns one 16-byte vector of channels and walks a block of tokens, keeping
// the last K - 1 inputs in registers; a warp covers 32 consecutive vectors of one token row.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;
constexpr int kConvTokens = 64;   // tokens per block (K - 1 extra rows read at the block start)

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16* p, float* f) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(h[e]);
    }
    __device__ static void store(__nv_bfloat16* p, const float* f) {
        uint4 u;
        __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __float2bfloat16_rn(f[e]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const float* p, float* f) {
        const float4 u = *reinterpret_cast<const float4*>(p);
        f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
    }
    __device__ static void store(float* p, const float* f) { *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]); }
};

// Sequence containing token t (largest i with start_i <= t, sequences sorted by start).
__device__ __forceinline__ int seq_of(const int32_t* cu, int nseq, int T_len, long long t) {
    int lo = 0, hi = nseq - 1, best = 0;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        long long a, b;
        seq_range(cu, mid, T_len, a, b);
        if (a <= t) { best = mid; lo = mid + 1; } else { hi = mid - 1; }
    }
    return best;
}

// Input vector of position p for sequence s starting at s0: x itself, or the cached input of the
// sequence (zeros without a cache) for the K-1 positions before its start.
template <typename T, int K>
__device__ __forceinline__ void load_input(const T* x, long long x_stride, const T* cache_in, int s, long long s0,
                                           long long p, int C, int c0, float (&f)[Vec<T>::N]) {
    if (p >= s0) {
        Vec<T>::load(x + p * x_stride + c0, f);
    } else {
#pragma unroll
        for (int e = 0; e < Vec<T>::N; ++e) f[e] = 0.f;
        if (cache_in) Vec<T>::load(cache_in + ((size_t)s * (K - 1) + (K - 1 - (s0 - p))) * C + c0, f);
    }
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads)
conv_fwd_kernel(const T* __restrict__ x, long long x_stride, const float* __restrict__ w,
                const T* __restrict__ cache_in, T* __restrict__ y, T* __restrict__ cache_out,
                const int32_t* __restrict__ cu, int nseq, int T_len, long long Ttot, int C) {
    constexpr int V = Vec<T>::N;
    const int vec = blockIdx.x * blockDim.x + threadIdx.x;
    if (vec * V >= C) return;
    const int c0 = vec * V;
    float wr[K][V];
#pragma unroll
    for (int e = 0; e < V; ++e)
#pragma unroll
        for (int i = 0; i < K; ++i) wr[i][e] = w[(size_t)(c0 + e) * K + i];

    // sequences without tokens pass their cache through (done once, by the first token block)
    if (blockIdx.y == 0 && cache_out) {
        for (int s = 0; s < nseq; ++s) {
            long long a, b;
            seq_range(cu, s, T_len, a, b);
            if (b > a) continue;
            for (int i = 0; i < K - 1; ++i) {
                float f[V];
                load_input<T, K>(x, x_stride, cache_in, s, a, a - (K - 1) + i, C, c0, f);
                Vec<T>::store(cache_out + ((size_t)s * (K - 1) + i) * C + c0, f);
            }
        }
    }
    for (long long tb = blockIdx.y; tb * kConvTokens < Ttot; tb += gridDim.y) {
        const long long t_end = min(Ttot, (tb + 1) * kConvTokens);
        long long t = tb * kConvTokens;
        while (t < t_end) {   // one segment per sequence the token block touches
            const int s = seq_of(cu, nseq, T_len, t);
            long long s0, s1;
            seq_range(cu, s, T_len, s0, s1);
            float hist[K][V];   // hist[K-1] = current token, hist[0] = oldest
#pragma unroll
            for (int i = 0; i < K - 1; ++i)
                load_input<T, K>(x, x_stride, cache_in, s, s0, t - (K - 1) + i, C, c0, hist[i]);
            const long long seg_end = min(t_end, s1);
#pragma unroll 4
            for (; t < seg_end; ++t) {
                Vec<T>::load(x + t * x_stride + c0, hist[K - 1]);
                float out[V];
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < K; ++i) acc = fmaf(wr[i][e], hist[i][e], acc);
                    out[e] = silu_f(acc);
                }
                Vec<T>::store(y + t * C + c0, out);
#pragma unroll
                for (int i = 0; i < K - 1; ++i)
#pragma unroll
                    for (int e = 0; e < V; ++e) hist[i][e] = hist[i + 1][e];
            }
            if (cache_out && seg_end == s1) {   // the sequence ended here: keep its last K - 1 inputs
#pragma unroll
                for (int i = 0; i < K - 1; ++i) Vec<T>::store(cache_out + ((size_t)s * (K - 1) + i) * C + c0, hist[i]);
            }
        }
    }
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvThreads)
conv_step_kernel(const T* __restrict__ x, long long x_stride, const float* __restrict__ w, T* __restrict__ cache,
                 T* __restrict__ y, int N, int C) {
    constexpr int V = Vec<T>::N;
    const int vec = blockIdx.x * blockDim.x + threadIdx.x;
    if (vec * V >= C) return;
    const int c0 = vec * V;
    for (size_t n = blockIdx.y; n < (size_t)N; n += gridDim.y) {
        float hist[K][V];
#pragma unroll
        for (int i = 0; i < K - 1; ++i) Vec<T>::load(cache + (n * (K - 1) + i) * C + c0, hist[i]);
        Vec<T>::load(x + (long long)n * x_stride + c0, hist[K - 1]);
        float out[V];
#pragma unroll
        for (int e = 0; e < V; ++e) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < K; ++i) acc = fmaf(w[(size_t)(c0 + e) * K + i], hist[i][e], acc);
            out[e] = silu_f(acc);
        }
        Vec<T>::store(y + n * C + c0, out);
#pragma unroll
        for (int i = 1; i < K; ++i) Vec<T>::store(cache + (n * (K - 1) + (i - 1)) * C + c0, hist[i]);
    }
}

// Threads per block: the channel vectors of one row, rounded up to whole warps, at most kConvThreads.
template <typename T>
int conv_threads(int C) {
    const int vecs = C / Vec<T>::N;
    return min(kConvThreads, (vecs + 31) / 32 * 32);
}

template <typename T, int K>
cudaError_t fwd_typed(const ConvArgs& a) {
    const long long Ttot = a.packed ? (long long)a.T : (long long)a.B * a.T;
    const int vecs = a.C / Vec<T>::N, threads = conv_threads<T>(a.C);
    const dim3 grid((unsigned)((vecs + threads - 1) / threads),
                    (unsigned)min(65535LL, max(1LL, (Ttot + kConvTokens - 1) / kConvTokens)));
    conv_fwd_kernel<T, K><<<grid, threads, 0, a.stream>>>(
        static_cast<const T*>(a.x), a.x_stride, a.w, static_cast<const T*>(a.cache_in), static_cast<T*>(a.y),
        static_cast<T*>(a.cache_out), a.cu_seqlens, a.num_seqs, a.T, Ttot, a.C);
    return cudaGetLastError();
}

template <typename T, int K>
cudaError_t step_typed(const ConvArgs& a) {
    const int vecs = a.C / Vec<T>::N, threads = conv_threads<T>(a.C);
    const dim3 grid((unsigned)((vecs + threads - 1) / threads), (unsigned)min(65535, a.B));
    conv_step_kernel<T, K><<<grid, threads, 0, a.stream>>>(static_cast<const T*>(a.x), a.x_stride, a.w,
                                                         static_cast<T*>(a.cache_out), static_cast<T*>(a.y),
                                                         a.B, a.C);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const ConvArgs& a, bool step) {
    switch (a.K) {
        case 1: return step ? step_typed<T, 1>(a) : fwd_typed<T, 1>(a);
        case 2: return step ? step_typed<T, 2>(a) : fwd_typed<T, 2>(a);
        case 3: return step ? step_typed<T, 3>(a) : fwd_typed<T, 3>(a);
        case 4: return step ? step_typed<T, 4>(a) : fwd_typed<T, 4>(a);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_conv_fwd(const ConvArgs& a) {
    return a.dtype == GDN_BF16 ? dispatch<__nv_bfloat16>(a, false) : dispatch<float>(a, false);
}

cudaError_t launch_conv_step(const ConvArgs& a) {
    if (a.B == 0) return cudaSuccess;
    return a.dtype == GDN_BF16 ? dispatch<__nv_bfloat16>(a, true) : dispatch<float>(a, true);
}

}  // namespace gdn
