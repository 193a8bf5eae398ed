// Depthwise causal short convolution + SiLU ("Transformer by Hand, ch. 7", listing
// "qwen/deltanet.py": conv1d(groups = channels, kernel K, padding K - 1) cut to the first T outputs,
// then SiLU; the parts table: each channel mixes only its own last few tokens; the learn-llm page:
// at inference the layer keeps the last K - 1 inputs of every sequence as a cache):
//     y[t, c] = silu( sum_{i=0}^{K-1} w[c, i] * x[t - (K - 1) + i, c] )
// with x before a sequence's first token taken from that sequence's cache (or zero).
//
// Memory bound (2 bytes read and written per element, ~10 instructions).  Forward pass: a persistent
// grid of two CTAs per SM walks tiles of 64 tokens x 512 bytes of channels.  A producer warp streams
// each tile plus its K - 1 halo rows into a 3-stage shared-memory ring with one bulk copy per token
// row (mbarrier completion); eight consumer warps each take a run of 8 tokens across the tile's 32
// channel vectors of 16 bytes, slide the K-row window in registers, and store 512-byte rows of y.
// Decode step: one thread per 16-byte channel vector of one sequence, cache shifted in place.
#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kRowBytes = 512;                    // channel slice of one tile row
constexpr int kTileTokens = 64;
constexpr int kHalo = 3;                          // rows kept before the tile (K - 1 <= 3)
constexpr int kStageRows = kTileTokens + kHalo;
constexpr int kStageBytes = kStageRows * kRowBytes;
constexpr int kStages = 3;
constexpr int kConsumerWarps = 8;                 // one run of kTileTokens / 8 tokens each
constexpr int kRunTokens = kTileTokens / kConsumerWarps;
constexpr int kFwdThreads = 32 * (kConsumerWarps + 1);
constexpr int kBarOffset = kStages * kStageBytes;
constexpr int kFwdSmem = kBarOffset + 2 * kStages * 8 + 16;
constexpr int kStepThreads = 128;
static_assert(kRowBytes / 16 == 32, "a warp covers one tile row with 16-byte vectors");
static_assert(2 * kFwdSmem + 2048 <= 228 * 1024, "two CTAs per SM");

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void unpack(const uint4& u, float* f) {
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(h[e]);
    }
    __device__ static uint4 pack(const float* f) {
        uint4 u;
        __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __float2bfloat16_rn(f[e]);
        return u;
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void unpack(const uint4& u, float* f) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
    __device__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float* f) { Vec<T>::unpack(*reinterpret_cast<const uint4*>(p), f); }
template <typename T>
__device__ __forceinline__ void store_vec(T* p, const float* f) { *reinterpret_cast<uint4*>(p) = Vec<T>::pack(f); }

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

// Cached input j (0 = oldest of the K - 1) of sequence s, zeros without a cache.
template <typename T, int K>
__device__ __forceinline__ void load_cached(const T* cache_in, int s, int j, int C, int c0, float (&f)[Vec<T>::N]) {
    if (cache_in) {
        load_vec(cache_in + ((size_t)s * (K - 1) + j) * C + c0, f);
    } else {
#pragma unroll
        for (int e = 0; e < Vec<T>::N; ++e) f[e] = 0.f;
    }
}

// SiLU for the output type: exact (ex2 + reciprocal) for fp32 outputs; for bf16 outputs one MUFU op,
// silu(z) = z/2 * (1 + tanh(z/2)) with the hardware tanh (relative error ~2^-11, below the 2^-9
// rounding of a bf16 result), which halves the special-function work that otherwise caps the kernel.
template <typename T>
__device__ __forceinline__ float silu_out(float z) { return silu_f(z); }
template <>
__device__ __forceinline__ float silu_out<__nv_bfloat16>(float z) {
    const float h = 0.5f * z;
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(h));
    return fmaf(h, th, h);
}

template <typename T, int K>
__device__ __forceinline__ void conv_out(const float (&wr)[K][Vec<T>::N], const float (&hist)[K][Vec<T>::N],
                                         float (&out)[Vec<T>::N]) {
#pragma unroll
    for (int e = 0; e < Vec<T>::N; ++e) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < K; ++i) acc = fmaf(wr[i][e], hist[i][e], acc);
        out[e] = silu_out<T>(acc);
    }
}

template <typename T, int K>
__global__ void __launch_bounds__(kFwdThreads, 2)
conv_fwd_kernel(const T* __restrict__ x, long long x_stride, const float* __restrict__ w,
                const T* __restrict__ cache_in, T* __restrict__ y, T* __restrict__ cache_out,
                const int32_t* __restrict__ cu, int nseq, int T_len, long long Ttot, int C, unsigned* status) {
    constexpr int V = Vec<T>::N;
    constexpr int CW = kRowBytes / (int)sizeof(T);      // channels per tile
    extern __shared__ __align__(1024) uint8_t sm[];
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar_full = sbase + kBarOffset, bar_empty = bar_full + 8 * kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kBarOffset + 16 * kStages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int n_cg = (C + CW - 1) / CW;
    const long long n_tt = (Ttot + kTileTokens - 1) / kTileTokens;
    const long long tiles = (long long)n_cg * n_tt;
    // contiguous tile range of this CTA (channel group major, so weights change rarely)
    const long long first = tiles * blockIdx.x / gridDim.x, last = tiles * (blockIdx.x + 1) / gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, kConsumerWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer: one bulk copy per token row of each tile
        for (long long i = first; i < last; ++i) {
            const int st = (int)((i - first) % kStages);
            const uint32_t ph = (uint32_t)(((i - first) / kStages) & 1);
            mbar_wait_bounded(bar_empty + 8 * st, ph ^ 1u, abort_flag, status, kStatusTimeout, kWaitLimitNs);
            const int cg = (int)(i / n_tt);
            const long long t0 = (i % n_tt) * kTileTokens;
            const long long r_lo = max(0LL, t0 - kHalo), r_hi = min(Ttot, t0 + kTileTokens);
            const uint32_t rb = (uint32_t)(min(CW, C - cg * CW) * (int)sizeof(T));
            if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * st, (uint32_t)(r_hi - r_lo) * rb);
            __syncwarp();
            for (long long r = r_lo + lane; r < r_hi; r += 32)
                bulk_g2s(sbase + st * kStageBytes + (uint32_t)(r - (t0 - kHalo)) * kRowBytes,
                         x + r * x_stride + (size_t)cg * CW, rb, bar_full + 8 * st);
        }
        // no copy of this CTA may still be writing shared memory when it exits
        if (lane == 0) {
            const long long n = last - first;
            for (long long j = max(0LL, n - kStages); j < n; ++j)
                mbar_wait_drain(bar_full + 8 * (uint32_t)(j % kStages), (uint32_t)((j / kStages) & 1), kWaitLimitNs);
        }
        return;
    }

    // ---------------- consumers
    if (blockIdx.x == 0 && cache_out) {
        // sequences without tokens pass their cache through
        for (int s = 0; s < nseq; ++s) {
            long long a, b;
            seq_range(cu, s, T_len, a, b);
            if (b > a) continue;
            for (int idx = threadIdx.x; idx < (K - 1) * (C / V); idx += 32 * kConsumerWarps) {
                const int j = idx / (C / V), c0 = (idx % (C / V)) * V;
                float f[V];
                load_cached<T, K>(cache_in, s, j, C, c0, f);
                store_vec(cache_out + ((size_t)s * (K - 1) + j) * C + c0, f);
            }
        }
    }
    float wr[K][V];
    int cg_loaded = -1;
    for (long long i = first; i < last; ++i) {
        const int st = (int)((i - first) % kStages);
        const uint32_t ph = (uint32_t)(((i - first) / kStages) & 1);
        const int cg = (int)(i / n_tt);
        const long long t0 = (i % n_tt) * kTileTokens;
        const int c0 = cg * CW + lane * V;
        const bool active = c0 < C;
        if (cg != cg_loaded && active) {
#pragma unroll
            for (int e = 0; e < V; ++e)
#pragma unroll
                for (int k = 0; k < K; ++k) wr[k][e] = __ldg(w + (size_t)(c0 + e) * K + k);
            cg_loaded = cg;
        }
        mbar_wait_bounded(bar_full + 8 * st, ph, abort_flag, status, kStatusTimeout, kWaitLimitNs);
        const uint8_t* stage = sm + st * kStageBytes + lane * 16;
        const long long row0 = t0 - kHalo;   // token of stage row 0
        long long t = t0 + warp * kRunTokens;
        const long long t_end = min(Ttot, t + kRunTokens);
        const auto row = [&](long long tok) { return *reinterpret_cast<const uint4*>(stage + (tok - row0) * kRowBytes); };
        int s = 0;
        long long s0 = 0, s1 = 0;
        if (active && t < t_end) {
            s = seq_of(cu, nseq, T_len, t);
            seq_range(cu, s, T_len, s0, s1);
        }
        if (active && t_end - t == kRunTokens && s0 <= t - (K - 1) && t + kRunTokens <= s1) {
            // common case: a whole run inside one sequence with its history in the tile; fully
            // unrolled, so the window slides by renaming registers
            float hist[K][V];
#pragma unroll
            for (int k = 0; k < K - 1; ++k) Vec<T>::unpack(row(t - (K - 1) + k), hist[k]);
#pragma unroll
            for (int j = 0; j < kRunTokens; ++j) {
                Vec<T>::unpack(row(t + j), hist[K - 1]);
                float out[V];
                conv_out<T, K>(wr, hist, out);
                store_vec(y + (t + j) * C + c0, out);
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
#pragma unroll
                    for (int e = 0; e < V; ++e) hist[k][e] = hist[k + 1][e];
            }
            if (cache_out && t + kRunTokens == s1) {
#pragma unroll
                for (int k = 0; k < K - 1; ++k) store_vec(cache_out + ((size_t)s * (K - 1) + k) * C + c0, hist[k]);
            }
            t = t_end;
        }
        while (active && t < t_end) {   // general case: one segment per sequence the run touches
            if (t >= s1) {
                s = seq_of(cu, nseq, T_len, t);
                seq_range(cu, s, T_len, s0, s1);
            }
            float hist[K][V];   // hist[K-1] = current token, hist[0] = oldest
#pragma unroll
            for (int k = 0; k < K - 1; ++k) {
                const long long src = t - (K - 1) + k;
                if (src >= s0)
                    Vec<T>::unpack(row(src), hist[k]);
                else
                    load_cached<T, K>(cache_in, s, (int)(K - 1 - (s0 - src)), C, c0, hist[k]);
            }
            const long long seg_end = min(t_end, s1);
#pragma unroll 1
            for (; t < seg_end; ++t) {
                Vec<T>::unpack(row(t), hist[K - 1]);
                float out[V];
                conv_out<T, K>(wr, hist, out);
                store_vec(y + t * C + c0, out);
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
#pragma unroll
                    for (int e = 0; e < V; ++e) hist[k][e] = hist[k + 1][e];
            }
            if (cache_out && seg_end == s1) {   // the sequence ended here: keep its last K - 1 inputs
#pragma unroll
                for (int k = 0; k < K - 1; ++k) store_vec(cache_out + ((size_t)s * (K - 1) + k) * C + c0, hist[k]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }
}

template <typename T, int K>
__global__ void __launch_bounds__(kStepThreads)
conv_step_kernel(const T* __restrict__ x, long long x_stride, const float* __restrict__ w, T* __restrict__ cache,
                 T* __restrict__ y, int N, int C) {
    constexpr int V = Vec<T>::N;
    const int vec = blockIdx.x * blockDim.x + threadIdx.x;
    if (vec * V >= C) return;
    const int c0 = vec * V;
    float wr[K][V];
#pragma unroll
    for (int e = 0; e < V; ++e)
#pragma unroll
        for (int k = 0; k < K; ++k) wr[k][e] = __ldg(w + (size_t)(c0 + e) * K + k);
    for (size_t n = blockIdx.y; n < (size_t)N; n += gridDim.y) {
        float hist[K][V];
#pragma unroll
        for (int k = 0; k < K - 1; ++k) load_vec(cache + (n * (K - 1) + k) * C + c0, hist[k]);
        load_vec(x + (long long)n * x_stride + c0, hist[K - 1]);
        float out[V];
        conv_out<T, K>(wr, hist, out);
        store_vec(y + n * C + c0, out);
#pragma unroll
        for (int k = 1; k < K; ++k) store_vec(cache + (n * (K - 1) + (k - 1)) * C + c0, hist[k]);
    }
}

template <typename T, int K>
cudaError_t fwd_typed(const ConvArgs& a) {
    const long long Ttot = a.packed ? (long long)a.T : (long long)a.B * a.T;
    constexpr int CW = kRowBytes / (int)sizeof(T);
    const long long tiles = (long long)((a.C + CW - 1) / CW) * ((Ttot + kTileTokens - 1) / kTileTokens);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(conv_fwd_kernel<T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(conv_fwd_kernel<T, K>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    // at least one CTA: it also passes the caches of sequences without tokens through
    const unsigned grid = (unsigned)max(1LL, min(tiles, 2LL * sms));
    conv_fwd_kernel<T, K><<<grid, kFwdThreads, kFwdSmem, a.stream>>>(
        static_cast<const T*>(a.x), a.x_stride, a.w, static_cast<const T*>(a.cache_in), static_cast<T*>(a.y),
        static_cast<T*>(a.cache_out), a.cu_seqlens, a.num_seqs, a.T, Ttot, a.C, a.status);
    return cudaGetLastError();
}

template <typename T, int K>
cudaError_t step_typed(const ConvArgs& a) {
    const int vecs = a.C / Vec<T>::N;
    const int threads = min(kStepThreads, (vecs + 31) / 32 * 32);
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
