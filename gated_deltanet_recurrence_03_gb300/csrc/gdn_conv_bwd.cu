// Backward of the depthwise causal short convolution + SiLU ("Transformer by Hand, ch. 7", listing
// "qwen/deltanet.py": conv1d(groups = channels, kernel K, padding K - 1) cut to the first T outputs,
// then SiLU; the decode cache of the learn-llm "linear attention" page holds the last K - 1 inputs).
// With xp the inputs of a sequence padded on the left by its K - 1 cached inputs and
//     u_t = sum_{j<K} w[c, j] xp[t + j],   y_t = silu(u_t),   du_t = dy_t silu'(u_t),
// the gradients are
//     dxp[p] = sum_j w[c, j] du_{p - j}     (the input at p feeds the outputs p - j, j < K)
//     dw[c, j] = sum_t du_t xp[t + j]
// and the outgoing cache (the last K - 1 rows of xp) passes its gradient straight to those rows.
// One thread per (64-token slot of a sequence, 4-byte vector of channels): it slides a K-row window of
// x and a K-entry ring of du over its tokens plus K - 1 on each side, the raw rows loaded three ahead (the du of the next slot's first
// tokens are recomputed, so slots are independent), writes dx of its own tokens (and of the cached
// inputs in a sequence's first slot) and its share of dw; column_sum_kernel adds the slots' shares in a
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

// 4-byte vectors of channels (2 bf16 or 1 fp32): a warp covers 128 contiguous bytes of a row, and the
// per-thread state fits 64 registers, four blocks of 256 threads per SM (measured on the 8k layer's
// projection: 16-byte vectors 926 us, 8-byte 749-769 us, 4-byte 641 us, 4-byte at four blocks per SM
// 519-521 us; five or more blocks per SM spill and run slower).
constexpr int kVecBytes = 4;
constexpr int kMinBlocks = 4;
constexpr int kPrefetch = 3;   // rows of x and dy loaded ahead of the row being used

template <typename T>
struct V4 {
    static constexpr int N = kVecBytes / (int)sizeof(T);
    using Raw = uint32_t;
    __device__ static Raw raw(const T* p) { return *reinterpret_cast<const Raw*>(p); }
    __device__ static void unpack(const Raw& u, float* f) {
        const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int e = 0; e < N; ++e) f[e] = to_f32(h[e]);
    }
    __device__ static void load(const T* p, float* f) { unpack(raw(p), f); }
};

template <int N>
__device__ __forceinline__ void store_f32(float* p, const float (&f)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int e = 0; e < N; e += 4) *reinterpret_cast<float4*>(p + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
    } else if constexpr (N == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(f[0], f[1]);
    } else {
        static_assert(N == 1, "one, two or a multiple of four channels");
        p[0] = f[0];
    }
}

template <typename T, int K>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
conv_bwd_kernel(const T* __restrict__ x, long long xs, const float* __restrict__ w, const T* __restrict__ cache_in,
                const T* __restrict__ dy, const T* __restrict__ dco, float* __restrict__ dx, float* __restrict__ dcache,
                float* __restrict__ partial, const int32_t* __restrict__ cu, int nseq, int T_len, int C,
                long long slots) {
    constexpr int VEC = V4<T>::N;
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
    // the raw bytes of the x row (an input, a cached input before the sequence, or zero past its end) and
    // of the dy row (zero outside this slot's tokens and halo, and past the sequence) of token tt
    using Raw = typename V4<T>::Raw;
    const auto fetch = [&](long long tt, Raw& rx, Raw& rd) {
        rx = 0u;
        rd = 0u;
        if (tt < s1) {
            if (tt >= s0)
                rx = V4<T>::raw(x + tt * xs + c0);
            else if (cache_in)
                rx = V4<T>::raw(cache_in + ((size_t)seq * (K - 1) + (size_t)(tt - s0 + K - 1)) * C + c0);
            if (tt >= t0) rd = V4<T>::raw(dy + tt * (long long)C + c0);
        }
    };
    float xw[K][VEC], dr[K][VEC];   // x rows t - K + 1 .. t (oldest first); du_{t - K + 1} .. du_t
#pragma unroll
    for (int j = 0; j < K; ++j)
#pragma unroll
        for (int e = 0; e < VEC; ++e) xw[j][e] = dr[j][e] = 0.f;
    const long long t_begin = t0 - (K - 1), t_end = t0 + n + K - 1;   // last du needed: token t0 + n + K - 2
    Raw qx[kPrefetch], qd[kPrefetch];   // rows t .. t + kPrefetch - 1, loaded ahead
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i) fetch(t_begin + i < t_end ? t_begin + i : s1, qx[i], qd[i]);
    for (long long t = t_begin; t < t_end; ++t) {
        const Raw rx = qx[0], rd = qd[0];
#pragma unroll
        for (int i = 0; i + 1 < kPrefetch; ++i) {
            qx[i] = qx[i + 1];
            qd[i] = qd[i + 1];
        }
        fetch(t + kPrefetch < t_end ? t + kPrefetch : s1, qx[kPrefetch - 1], qd[kPrefetch - 1]);
#pragma unroll
        for (int j = 0; j + 1 < K; ++j)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                xw[j][e] = xw[j + 1][e];
                dr[j][e] = dr[j + 1][e];
            }
        V4<T>::unpack(rx, xw[K - 1]);
        float* d = dr[K - 1];
        if (t >= t0 && t < s1) {   // du_t = dy_t silu'(u_t); this slot's own tokens add to dw
            float g[VEC];
            V4<T>::unpack(rd, g);
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
                float acc_x = 0.f;
#pragma unroll
                for (int j = 0; j < K; ++j) acc_x = fmaf(wv[e][j], dr[K - 1 - j][e], acc_x);
                gx[e] = acc_x;
            }
            if (dco && p >= s1 - (K - 1)) {   // the outgoing cache holds this input
                float gc[VEC];
                V4<T>::load(dco + ((size_t)seq * (K - 1) + (size_t)(p - (s1 - (K - 1)))) * C + c0, gc);
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

long long conv_slots(const ConvArgs& a) {
    const long long ttot = a.packed ? (long long)a.T : (long long)a.B * a.T;
    return (ttot + kSlot - 1) / kSlot + a.num_seqs;
}

template <typename T, int K>
cudaError_t launch_k(const ConvArgs& a, const void* dy, const void* dco, float* dx, float* dw, float* dcache,
                     float* partial) {
    constexpr int VEC = V4<T>::N;
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
        column_sum_kernel<<<(CK + 31) / 32, kColSumThreads, 0, a.stream>>>(partial, slots, CK, dw);
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
