// Depthwise causal short convolution + SiLU ("Transformer by Hand, ch. 7", listing
// "qwen/deltanet.py": conv1d(groups = channels, kernel K, padding K - 1) cut to the first T outputs,
// then SiLU; the parts table: each channel mixes only its own last few tokens; the learn-llm page:
// at inference the layer keeps the last K - 1 inputs of every sequence as a cache):
//     y[t, c] = silu( sum_{i=0}^{K-1} w[c, i] * x[t - (K - 1) + i, c] )
// with x before a sequence's first token taken from that sequence's cache (or zero).
//
// Memory bound (2 bytes read and written per element, ~6 instructions).  Forward pass: a persistent
// grid of one CTA per SM walks tiles of 128 tokens x 512 bytes of channels, in token-major order.
// Each tile plus its K - 1 halo rows arrives in a 3-stage shared-memory ring by one 2-D TMA copy
// (rows before the first token or past the last come back as zeros; mbarrier completion), issued by
// one thread once all eight warps have released the stage.  Each warp takes a run of 16 tokens
// across the tile's 32 channel vectors of 16 bytes, slides the K-row window in registers (packed
// fp32x2 arithmetic) and streams 512-byte rows of y out.
// Decode step: one thread per 16-byte channel vector of one sequence, cache shifted in place.
// Both can split their output by channel into up to three contiguous tensors (the q, k and v slices
// of the packed projection the layer convolves in one pass), whatever the split, one launch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kRowBytes = 512;                    // channel slice of one tile row
constexpr int kTileTokens = 128;
constexpr int kHalo = 3;                          // rows kept before the tile (K - 1 <= 3)
constexpr int kStageRows = kTileTokens + kHalo;
constexpr int kStageBytes = kStageRows * kRowBytes;
constexpr int kStages = 3;
constexpr int kConsumerWarps = 8;                 // one run of kTileTokens / 8 tokens each
constexpr int kRunTokens = kTileTokens / kConsumerWarps;
constexpr int kFwdThreads = 32 * kConsumerWarps;   // lane 0 of warp 0 also issues the tile copies
constexpr int kBarOffset = kStages * kStageBytes;
constexpr int kFwdSmem = kBarOffset + 2 * kStages * 8 + 16;
constexpr int kStepThreads = 128;
static_assert(kRowBytes / 16 == 32, "a warp covers one tile row with 16-byte vectors");
static_assert(kFwdSmem <= 227 * 1024, "one CTA per SM");

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    // channel pairs: a bf16 widens to fp32 by a 16-bit shift
    __device__ static void unpack2(const uint4& u, float2* f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) f[p] = make_float2(__uint_as_float(w[p] << 16), __uint_as_float(w[p] & 0xffff0000u));
    }
    __device__ static uint4 pack2(const float2* f) {
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const __nv_bfloat162 h = __float22bfloat162_rn(f[p]);
            w[p] = *reinterpret_cast<const uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void unpack2(const uint4& u, float2* f) {
        f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
        f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
    __device__ static uint4 pack2(const float2* f) {
        return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x), __float_as_uint(f[1].y));
    }
};

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float2* f) { Vec<T>::unpack2(*reinterpret_cast<const uint4*>(p), f); }
template <typename T>
__device__ __forceinline__ void store_vec(T* p, const float2* f) { __stcs(reinterpret_cast<uint4*>(p), Vec<T>::pack2(f)); }

// Where the outputs of one 16-byte channel vector go: y (channels [0, c1)), y_k ([c1, c2)) or y_v
// ([c2, C)), each a dense [rows, width] tensor; without a split, y holds all C channels.
template <typename T>
struct OutSplit {
    T* y;
    T* y_k;
    T* y_v;
    int c1, c2, C;
    __device__ __forceinline__ void route(int c0, T*& base, int& width, int& col) const {
        if (!y_k || c0 < c1) { base = y; width = y_k ? c1 : C; col = c0; }
        else if (c0 < c2) { base = y_k; width = c2 - c1; col = c0 - c1; }
        else { base = y_v; width = C - c2; col = c0 - c2; }
    }
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

// Cached input j (0 = oldest of the K - 1) of sequence s, zeros without a cache.
template <typename T, int K>
__device__ __forceinline__ void load_cached(const T* cache_in, int s, int j, int C, int c0, float2 (&f)[Vec<T>::N / 2]) {
    if (cache_in) {
        load_vec(cache_in + ((size_t)s * (K - 1) + j) * C + c0, f);
    } else {
#pragma unroll
        for (int p = 0; p < Vec<T>::N / 2; ++p) f[p] = make_float2(0.f, 0.f);
    }
}

// SiLU of a channel pair for the output type: exact (ex2 + reciprocal) for fp32 outputs; for bf16
// outputs one MUFU op per value, silu(z) = z/2 * (1 + tanh(z/2)) with the hardware tanh (relative
// error ~2^-11, below the 2^-9 rounding of a bf16 result), which halves the special-function work
// that otherwise caps the kernel.
template <typename T>
__device__ __forceinline__ float2 silu_out2(float2 z) { return make_float2(silu_f(z.x), silu_f(z.y)); }
template <>
__device__ __forceinline__ float2 silu_out2<__nv_bfloat16>(float2 z) {
    const float2 h = __fmul2_rn(z, make_float2(0.5f, 0.5f));
    float2 th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th.x) : "f"(h.x));
    asm("tanh.approx.f32 %0, %1;" : "=f"(th.y) : "f"(h.y));
    return __ffma2_rn(h, th, h);
}

// Channel pairs of one 16-byte vector; the K taps as packed fp32x2 multiply-adds, oldest first.
template <typename T, int K>
__device__ __forceinline__ void conv_out(const float2 (&wr)[K][Vec<T>::N / 2], const float2 (&hist)[K][Vec<T>::N / 2],
                                         float2 (&out)[Vec<T>::N / 2]) {
#pragma unroll
    for (int p = 0; p < Vec<T>::N / 2; ++p) {
        float2 acc = __fmul2_rn(wr[0][p], hist[0][p]);
#pragma unroll
        for (int i = 1; i < K; ++i) acc = __ffma2_rn(wr[i][p], hist[i][p], acc);
        out[p] = silu_out2<T>(acc);
    }
}

// The K taps of channels c0 .. c0 + V - 1 as channel pairs: one vector load per channel when K is 2 or 4
// and the rows are aligned (uniform over the grid), scalar loads otherwise.
template <typename T, int K>
__device__ __forceinline__ void load_taps(const float* __restrict__ w, int c0, bool vec_ok,
                                          float2 (&wr)[K][Vec<T>::N / 2]) {
    constexpr int P = Vec<T>::N / 2;
    float t[2 * P][K];
#pragma unroll
    for (int e = 0; e < 2 * P; ++e) {
        const float* src = w + (size_t)(c0 + e) * K;
        if constexpr (K == 4) {
            if (vec_ok) {
                const float4 f = __ldg(reinterpret_cast<const float4*>(src));
                t[e][0] = f.x; t[e][1] = f.y; t[e][2] = f.z; t[e][3] = f.w;
                continue;
            }
        } else if constexpr (K == 2) {
            if (vec_ok) {
                const float2 f = __ldg(reinterpret_cast<const float2*>(src));
                t[e][0] = f.x; t[e][1] = f.y;
                continue;
            }
        }
#pragma unroll
        for (int k = 0; k < K; ++k) t[e][k] = __ldg(src + k);
    }
#pragma unroll
    for (int p = 0; p < P; ++p)
#pragma unroll
        for (int k = 0; k < K; ++k) wr[k][p] = make_float2(t[2 * p][k], t[2 * p + 1][k]);
}

template <typename T, int K>
__global__ void __launch_bounds__(kFwdThreads, 1)
conv_fwd_kernel(const __grid_constant__ CUtensorMap xmap, const float* __restrict__ w,
                const T* __restrict__ cache_in, const OutSplit<T> ys, T* __restrict__ cache_out,
                const int32_t* __restrict__ cu, int nseq, int T_len, long long Ttot, int C, unsigned* status) {
    constexpr int V = Vec<T>::N, P = V / 2;
    constexpr int CW = kRowBytes / (int)sizeof(T);      // channels per tile
    extern __shared__ __align__(1024) uint8_t sm[];
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bar_full = sbase + kBarOffset, bar_empty = bar_full + 8 * kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kBarOffset + 16 * kStages);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int n_cg = (C + CW - 1) / CW;
    const long long n_tt = (Ttot + kTileTokens - 1) / kTileTokens;
    const long long tiles = (long long)n_cg * n_tt;
    // tiles in token-major order (tile i = token tile i / n_cg, channel group i % n_cg), CTA b taking
    // b, b + G, b + 2G, ...: the CTAs in flight together read whole token rows, and when G is a
    // multiple of n_cg each CTA keeps one channel group (and its weights) throughout
    const long long G = gridDim.x;
    const long long my_tiles = blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / G + 1 : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, kConsumerWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    // one 2-D TMA copy per tile: 67 rows x 512 bytes, row 0 = token t0 - kHalo
    const bool producer = threadIdx.x == 0;
    const auto issue = [&](long long n) {
        const long long i = blockIdx.x + n * G;
        const int st = (int)(n % kStages);
        mbar_arrive_expect_tx(bar_full + 8 * st, kStageBytes);
        tma_load_2d(sbase + st * kStageBytes, &xmap, (int)(i % n_cg) * CW, (int)((i / n_cg) * kTileTokens - kHalo),
                    bar_full + 8 * st);
    };
    if (producer)
        for (long long n = 0; n < min((long long)kStages, my_tiles); ++n) issue(n);

    // ---------------- consumers
    if (blockIdx.x == 0 && cache_out) {
        // sequences without tokens pass their cache through
        for (int s = 0; s < nseq; ++s) {
            long long a, b;
            seq_range(cu, s, T_len, a, b);
            if (b > a) continue;
            for (int idx = threadIdx.x; idx < (K - 1) * (C / V); idx += kFwdThreads) {
                const int j = idx / (C / V), c0 = (idx % (C / V)) * V;
                float2 f[P];
                load_cached<T, K>(cache_in, s, j, C, c0, f);
                store_vec(cache_out + ((size_t)s * (K - 1) + j) * C + c0, f);
            }
        }
    }
    float2 wr[K][P];
    int cg_loaded = -1;
    for (long long n = 0; n < my_tiles; ++n) {
        const long long i = blockIdx.x + n * G;
        const int st = (int)(n % kStages);
        const uint32_t ph = (uint32_t)((n / kStages) & 1);
        const int cg = (int)(i % n_cg);
        const long long t0 = (i / n_cg) * kTileTokens;
        const int c0 = cg * CW + lane * V;
        const bool active = c0 < C;
        T* yb;
        int yw, yc;
        ys.route(c0, yb, yw, yc);
        T* __restrict__ y = yb + yc;   // token t of this vector at y[t * yw]
        if (cg != cg_loaded && active) {
            load_taps<T, K>(w, c0, (reinterpret_cast<uintptr_t>(w) % (K * sizeof(float))) == 0, wr);
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
            float2 hist[K][P];
#pragma unroll
            for (int k = 0; k < K - 1; ++k) Vec<T>::unpack2(row(t - (K - 1) + k), hist[k]);
#pragma unroll
            for (int j = 0; j < kRunTokens; ++j) {
                Vec<T>::unpack2(row(t + j), hist[K - 1]);
                float2 out[P];
                conv_out<T, K>(wr, hist, out);
                store_vec(y + (t + j) * yw, out);
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
#pragma unroll
                    for (int p = 0; p < P; ++p) hist[k][p] = hist[k + 1][p];
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
            float2 hist[K][P];   // hist[K-1] = current token, hist[0] = oldest
#pragma unroll
            for (int k = 0; k < K - 1; ++k) {
                const long long src = t - (K - 1) + k;
                if (src >= s0)
                    Vec<T>::unpack2(row(src), hist[k]);
                else
                    load_cached<T, K>(cache_in, s, (int)(K - 1 - (s0 - src)), C, c0, hist[k]);
            }
            const long long seg_end = min(t_end, s1);
#pragma unroll 1
            for (; t < seg_end; ++t) {
                Vec<T>::unpack2(row(t), hist[K - 1]);
                float2 out[P];
                conv_out<T, K>(wr, hist, out);
                store_vec(y + t * yw, out);
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
#pragma unroll
                    for (int p = 0; p < P; ++p) hist[k][p] = hist[k + 1][p];
            }
            if (cache_out && seg_end == s1) {   // the sequence ended here: keep its last K - 1 inputs
#pragma unroll
                for (int k = 0; k < K - 1; ++k) store_vec(cache_out + ((size_t)s * (K - 1) + k) * C + c0, hist[k]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * st);
        if (producer && n + kStages < my_tiles) {   // refill the stage once every warp has left it
            mbar_wait_bounded(bar_empty + 8 * st, ph, abort_flag, status, kStatusTimeout, kWaitLimitNs);
            issue(n + kStages);
        }
    }
    // no copy of this CTA may still be writing shared memory when it exits
    if (producer)
        for (long long j = max(0LL, my_tiles - kStages); j < my_tiles; ++j)
            mbar_wait_drain(bar_full + 8 * (uint32_t)(j % kStages), (uint32_t)((j / kStages) & 1), kWaitLimitNs);
}

// One thread per 16-byte channel vector and block of kStepRows sequences: the weights are loaded
// once and reused.  Every row's cache and input vectors are loaded before any row is written (the
// cache is updated in place, so loads placed after a row's stores could not be hoisted above them),
// which keeps 4 K 16-byte loads of each thread in flight together.
constexpr int kStepRows = 4;

template <typename T, int K>
__global__ void __launch_bounds__(kStepThreads)
conv_step_kernel(const T* __restrict__ x, long long x_stride, const float* __restrict__ w, T* __restrict__ cache,
                 const OutSplit<T> ys, int N, int C) {
    constexpr int V = Vec<T>::N, P = V / 2;
    const int vec = blockIdx.x * blockDim.x + threadIdx.x;
    if (vec * V >= C) return;
    const int c0 = vec * V;
    T* yb;
    int yw, yc;
    ys.route(c0, yb, yw, yc);
    float2 wr[K][P];
    load_taps<T, K>(w, c0, (reinterpret_cast<uintptr_t>(w) % (K * sizeof(float))) == 0, wr);
    for (size_t n0 = (size_t)blockIdx.y * kStepRows; n0 < (size_t)N; n0 += (size_t)gridDim.y * kStepRows) {
        uint4 raw[kStepRows][K];   // the K - 1 cached inputs, oldest first, then this step's input
#pragma unroll
        for (int r = 0; r < kStepRows; ++r) {
            const size_t n = n0 + r;
            if (n < (size_t)N) {
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
                    raw[r][k] = *reinterpret_cast<const uint4*>(cache + (n * (K - 1) + k) * C + c0);
                raw[r][K - 1] = *reinterpret_cast<const uint4*>(x + (long long)n * x_stride + c0);
            } else {
#pragma unroll
                for (int k = 0; k < K; ++k) raw[r][k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int r = 0; r < kStepRows; ++r) {
            const size_t n = n0 + r;
            if (n >= (size_t)N) break;
            float2 hist[K][P];
#pragma unroll
            for (int k = 0; k < K; ++k) Vec<T>::unpack2(raw[r][k], hist[k]);
            float2 out[P];
            conv_out<T, K>(wr, hist, out);
            store_vec(yb + n * yw + yc, out);
#pragma unroll
            for (int k = 1; k < K; ++k) __stcs(reinterpret_cast<uint4*>(cache + (n * (K - 1) + (k - 1)) * C + c0), raw[r][k]);
        }
    }
}

template <typename T, int K>
cudaError_t fwd_typed(const ConvArgs& a) {
    const long long Ttot = a.packed ? (long long)a.T : (long long)a.B * a.T;
    constexpr int CW = kRowBytes / (int)sizeof(T);
    const long long n_cg = (a.C + CW - 1) / CW;
    const long long tiles = n_cg * ((Ttot + kTileTokens - 1) / kTileTokens);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(conv_fwd_kernel<T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(conv_fwd_kernel<T, K>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    // one CTA per SM, rounded down to a multiple of the channel groups when there are fewer groups
    // than CTAs (a grid of every SM, each CTA reloading its taps when its group changes, measured the
    // same on the 8192-channel projection: 0.101 ms); at least one CTA, which also passes the caches
    // of sequences without tokens through
    long long G = sms;
    if (n_cg <= G) G = G / n_cg * n_cg;
    const unsigned grid = (unsigned)max(1LL, min(tiles, G));
    // x as a 2-D tensor [Ttot rows, C channels] with a row pitch of x_stride elements; box of
    // kStageRows rows x CW channels, zero fill outside
    CUtensorMap xmap;
    memset(&xmap, 0, sizeof(xmap));
    if (tiles > 0) {
        if (Ttot > (1LL << 31) - 2 * kTileTokens) return cudaErrorInvalidValue;   // TMA coordinates are 32-bit
        auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
        if (!encode) return cudaErrorNotSupported;
        const cuuint64_t dims[2] = {(cuuint64_t)a.C, (cuuint64_t)Ttot};
        const cuuint64_t strides[1] = {(cuuint64_t)a.x_stride * sizeof(T)};
        const cuuint32_t box[2] = {(cuuint32_t)CW, (cuuint32_t)kStageRows};
        const cuuint32_t elem[2] = {1, 1};
        const CUresult r = encode(&xmap, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                  2, const_cast<void*>(a.x), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    const OutSplit<T> ys{static_cast<T*>(a.y), static_cast<T*>(a.y_k), static_cast<T*>(a.y_v), a.c1, a.c2, a.C};
    conv_fwd_kernel<T, K><<<grid, kFwdThreads, kFwdSmem, a.stream>>>(
        xmap, a.w, static_cast<const T*>(a.cache_in), ys, static_cast<T*>(a.cache_out), a.cu_seqlens, a.num_seqs,
        a.T, Ttot, a.C, a.status);
    return cudaGetLastError();
}

template <typename T, int K>
cudaError_t step_typed(const ConvArgs& a) {
    const int vecs = a.C / Vec<T>::N;
    const int threads = min(kStepThreads, (vecs + 31) / 32 * 32);
    const dim3 grid((unsigned)((vecs + threads - 1) / threads), (unsigned)min(65535, (a.B + kStepRows - 1) / kStepRows));
    const OutSplit<T> ys{static_cast<T*>(a.y), static_cast<T*>(a.y_k), static_cast<T*>(a.y_v), a.c1, a.c2, a.C};
    conv_step_kernel<T, K><<<grid, threads, 0, a.stream>>>(static_cast<const T*>(a.x), a.x_stride, a.w,
                                                         static_cast<T*>(a.cache_out), ys, a.B, a.C);
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
