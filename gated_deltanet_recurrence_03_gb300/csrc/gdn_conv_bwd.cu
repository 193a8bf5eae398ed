// Backward of the depthwise causal short convolution + SiLU ("Transformer by Hand, ch. 7", listing
// "qwen/deltanet.py": conv1d(groups = channels, kernel K, padding K - 1) cut to the first T outputs,
// then SiLU; the decode cache of the learn-llm "linear attention" page holds the last K - 1 inputs).
// With xp the inputs of a sequence padded on the left by its K - 1 cached inputs and
//     u_t = sum_{j<K} w[c, j] xp[t + j],   y_t = silu(u_t),   du_t = dy_t silu'(u_t),
// the gradients are
//     dxp[p] = sum_j w[c, j] du_{p - j}     (the input at p feeds the outputs p - j, j < K)
//     dw[c, j] = sum_t du_t xp[t + j]
// and the outgoing cache (the last K - 1 rows of xp) passes its gradient straight to those rows.
// One thread per (64-token slot of a sequence, 16-byte vector of channels): it slides a K-row window of
// x and a K-entry ring of du over its tokens plus K - 1 on each side (the du of the next slot's first
// tokens are recomputed, so slots are independent), writes dx of its own tokens (and of the cached
// inputs in a sequence's first slot) and its share of dw; a second kernel adds the slots' shares in a
// fixed order.
#include <algorithm>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kSlot = 64;          // tokens per slot
constexpr int kThreads = 256;

// Chunk c of sequence i occupies slot floor(start_i / 64) + i + c (no prefix sum needed).
__device__ bool conv_slot(const int32_t* cu, int nseq, int T_len, long long slot, int& seq, long long& t0, int& n) {
    int lo = 0, hi = nseq - 1, best = -1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        long long a, b;
        seq_range(cu, mid, T_len, a, b);
        if (a / kSlot + mid <= slot) {
            best = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    if (best < 0) return false;
    long long a, b;
    seq_range(cu, best, T_len, a, b);
    const long long c = slot - (a / kSlot + best);
    if (c < 0 || a + c * kSlot >= b) return false;
    seq = best;
    t0 = a + c * kSlot;
    n = (int)min((long long)kSlot, b - t0);
    return true;
}

template <typename T>
struct V16 {
    static constexpr int N = 16 / (int)sizeof(T);
    __device__ static void load(const T* p, float* f) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int e = 0; e < N; ++e) f[e] = to_f32(h[e]);
    }
};

template <int N>
__device__ __forceinline__ void store_f32(float* p, const float (&f)[N]) {
#pragma unroll
    for (int e = 0; e < N; e += 4) *reinterpret_cast<float4*>(p + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
}

template <typename T, int K>
__global__ void __launch_bounds__(kThreads)
conv_bwd_kernel(const T* __restrict__ x, long long xs, const float* __restrict__ w, const T* __restrict__ cache_in,
                const T* __restrict__ dy, const T* __restrict__ dco, float* __restrict__ dx, float* __restrict__ dcache,
                float* __restrict__ partial, const int32_t* __restrict__ cu, int nseq, int T_len, int C,
                long long slots) {
    constexpr int VEC = V16<T>::N;
    const int NV = C / VEC;
    const long long item = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (item >= slots * NV) return;
    const long long slot = item / NV;
    const int c0 = (int)(item % NV) * VEC;
    float acc[VEC][K];
#pragma unroll
    for (int e = 0; e < VEC; ++e)
#pragma unroll
        for (int j = 0; j < K; ++j) acc[e][j] = 0.f;
    float* part = partial ? partial + ((size_t)slot * C + c0) * K : nullptr;
    int seq, n;
    long long t0;
    if (!conv_slot(cu, nseq, T_len, slot, seq, t0, n)) {   // an unused slot adds nothing
        if (!part) return;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
#pragma unroll
            for (int j = 0; j < K; ++j) part[e * K + j] = 0.f;
        return;
    }
    long long s0, s1;
    seq_range(cu, seq, T_len, s0, s1);
    float wv[VEC][K];
#pragma unroll
    for (int e = 0; e < VEC; ++e)
#pragma unroll
        for (int j = 0; j < K; ++j) wv[e][j] = w[(size_t)(c0 + e) * K + j];
    float xw[K][VEC], dr[K][VEC];   // x rows t - K + 1 .. t (oldest first); du_{t - K + 1} .. du_t
#pragma unroll
    for (int j = 0; j < K; ++j)
#pragma unroll
        for (int e = 0; e < VEC; ++e) xw[j][e] = dr[j][e] = 0.f;
    const long long t_end = t0 + n + K - 1;   // last du needed is that of token t0 + n + K - 2
    for (long long t = t0 - (K - 1); t < t_end; ++t) {
#pragma unroll
        for (int j = 0; j + 1 < K; ++j)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                xw[j][e] = xw[j + 1][e];
                dr[j][e] = dr[j + 1][e];
            }
        // the newest window row: x, a cached input before the sequence, or nothing past its end
        float* xr = xw[K - 1];
        if (t >= s1) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) xr[e] = 0.f;
        } else if (t >= s0) {
            V16<T>::load(x + t * xs + c0, xr);
        } else if (cache_in) {
            V16<T>::load(cache_in + ((size_t)seq * (K - 1) + (size_t)(t - s0 + K - 1)) * C + c0, xr);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) xr[e] = 0.f;
        }
        float* d = dr[K - 1];
        if (t >= t0 && t < s1) {   // du_t = dy_t silu'(u_t); this slot's own tokens add to dw
            float g[VEC];
            V16<T>::load(dy + t * (long long)C + c0, g);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float u = 0.f;
#pragma unroll
                for (int j = 0; j < K; ++j) u = fmaf(wv[e][j], xw[j][e], u);
                const float sg = 1.f / (1.f + __expf(-u));
                d[e] = g[e] * sg * (1.f + u * (1.f - sg));
            }
            if (t < t0 + n) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
#pragma unroll
                    for (int j = 0; j < K; ++j) acc[e][j] = fmaf(d[e], xw[j][e], acc[e][j]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) d[e] = 0.f;
        }
        // the input at p = t - (K - 1) feeds the outputs p .. t: its gradient is complete now
        const long long p = t - (K - 1);
        const bool own = p >= t0 && p < t0 + n;
        const bool cached = K > 1 && dcache && t0 == s0 && p < s0 && p >= s0 - (K - 1);   // first slot: the cache
        if (own || cached) {
            float gx[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float a = 0.f;
#pragma unroll
                for (int j = 0; j < K; ++j) a = fmaf(wv[e][j], dr[K - 1 - j][e], a);
                gx[e] = a;
            }
            if (dco && p >= s1 - (K - 1)) {   // the outgoing cache holds this input
                float gc[VEC];
                V16<T>::load(dco + ((size_t)seq * (K - 1) + (size_t)(p - (s1 - (K - 1)))) * C + c0, gc);
#pragma unroll
                for (int e = 0; e < VEC; ++e) gx[e] += gc[e];
            }
            if (own)
                store_f32(dx + p * (long long)C + c0, gx);
            else
                store_f32(dcache + ((size_t)seq * (K - 1) + (size_t)(p - s0 + K - 1)) * C + c0, gx);
        }
    }
    if (!part) return;
#pragma unroll
    for (int e = 0; e < VEC; ++e)
#pragma unroll
        for (int j = 0; j < K; ++j) part[e * K + j] = acc[e][j];
}

// Sequences without tokens: the outgoing cache is the incoming one, so its gradient passes through.
template <typename T>
__global__ void conv_bwd_empty_kernel(const T* __restrict__ dco, float* __restrict__ dcache, const int32_t* __restrict__ cu,
                                      int nseq, int T_len, int C, int K) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long per = (long long)(K - 1) * C;
    if (i >= per * nseq) return;
    const int seq = (int)(i / per);
    long long a, b;
    seq_range(cu, seq, T_len, a, b);
    if (b > a) return;
    dcache[i] = dco ? to_f32(dco[i]) : 0.f;
}

// dw[c][j] = sum over slots (in order) of the slots' shares.
__global__ void conv_dw_reduce_kernel(const float* __restrict__ partial, long long slots, int CK, float* __restrict__ dw) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= CK) return;
    float t = 0.f;
    for (long long s = 0; s < slots; ++s) t += partial[(size_t)s * CK + i];
    dw[i] = t;
}

long long conv_slots(const ConvArgs& a) {
    const long long ttot = a.packed ? (long long)a.T : (long long)a.B * a.T;
    return (ttot + kSlot - 1) / kSlot + a.num_seqs;
}

template <typename T, int K>
cudaError_t launch_k(const ConvArgs& a, const void* dy, const void* dco, float* dx, float* dw, float* dcache,
                     float* partial) {
    constexpr int VEC = V16<T>::N;
    const long long slots = conv_slots(a);
    const long long items = slots * (a.C / VEC);
    const int T_len = a.T;
    const int32_t* cu = a.packed ? a.cu_seqlens : nullptr;
    if (items > 0)
        conv_bwd_kernel<T, K><<<(unsigned)((items + kThreads - 1) / kThreads), kThreads, 0, a.stream>>>(
            static_cast<const T*>(a.x), a.x_stride, a.w, static_cast<const T*>(a.cache_in), static_cast<const T*>(dy),
            static_cast<const T*>(dco), dx, dcache, partial, cu, a.num_seqs, T_len, a.C, slots);
    if (K > 1 && dcache) {
        const long long n = (long long)(K - 1) * a.C * a.num_seqs;
        conv_bwd_empty_kernel<T><<<(unsigned)((n + 255) / 256), 256, 0, a.stream>>>(static_cast<const T*>(dco), dcache, cu,
                                                                                   a.num_seqs, T_len, a.C, K);
    }
    if (dw) {
        const int CK = a.C * K;
        conv_dw_reduce_kernel<<<(CK + 255) / 256, 256, 0, a.stream>>>(partial, slots, CK, dw);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const ConvArgs& a, const void* dy, const void* dco, float* dx, float* dw, float* dcache,
                     float* partial) {
    switch (a.K) {
        case 1: return launch_k<T, 1>(a, dy, dco, dx, dw, dcache, partial);
        case 2: return launch_k<T, 2>(a, dy, dco, dx, dw, dcache, partial);
        case 3: return launch_k<T, 3>(a, dy, dco, dx, dw, dcache, partial);
        case 4: return launch_k<T, 4>(a, dy, dco, dx, dw, dcache, partial);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

size_t conv_bwd_workspace_bytes(int B, int T, int C, int K, int nseq, bool packed) {
    const long long ttot = packed ? (long long)T : (long long)B * T;
    const long long slots = (ttot + kSlot - 1) / kSlot + nseq;
    return (size_t)slots * C * K * sizeof(float);
}

cudaError_t launch_conv_bwd(const ConvArgs& a, const void* dy, const void* dco, float* dx, float* dw, float* dcache,
                            void* workspace) {
    float* partial = static_cast<float*>(workspace);
    return a.dtype == GDN_BF16 ? launch_t<__nv_bfloat16>(a, dy, dco, dx, dw, dcache, partial)
                               : launch_t<float>(a, dy, dco, dx, dw, dcache, partial);
}

}  // namespace gdn
