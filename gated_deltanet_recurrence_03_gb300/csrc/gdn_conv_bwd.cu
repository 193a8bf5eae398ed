// Backward of the depthwise causal short convolution + SiLU ("Transformer by Hand, ch. 7", listing
// "qwen/deltanet.py": conv1d(groups = channels, kernel K, padding K - 1) cut to the first T outputs,
// then SiLU; the decode cache of the learn-llm "linear attention" page holds the last K - 1 inputs).
// With xp the inputs of a sequence padded on the left by its K - 1 cached inputs and
//     u_t = sum_{j<K} w[c, j] xp[t + j],   y_t = silu(u_t),   du_t = dy_t silu'(u_t),
// the gradients are
//     dxp[p] = sum_j w[c, j] du_{p - j}     (the input at p feeds the outputs p - j, j < K)
//     dw[c, j] = sum_t du_t xp[t + j]
// and the outgoing cache (the last K - 1 rows of xp) passes its gradient straight to those rows.
// Each 64-token slot of a sequence (chunk c of sequence i in slot floor(start_i / 64) + i + c) is
// handled with its K - 1 tokens of halo on each side, so slots are independent; the slots' shares of dw
// are added by column_sum_kernel in a fixed order.
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

// One block of 256 threads per (64-token slot, block of channels of 256 bytes a row: 128 bf16 or 64 fp32):
//  1. the slot's x rows (its tokens with K - 1 before and after; cached inputs before the sequence, zeros
//     past it) and dy rows (its tokens and K - 1 after) are copied to shared memory with 16-byte loads,
//     whole rows per half-warp;
//  2. du = dy silu'(u) for the slot's tokens and the K - 1 after, each thread a channel pair and every
//     NG-th token, into shared memory in fp32; the thread's own tokens add to its taps' sums;
//  3. dx of the slot's tokens (and of the cached inputs in a sequence's first slot) from K neighbouring
//     du rows, written as whole fp32 rows;
//  4. the taps' sums of the token groups are added in a fixed order into the slot's share of dw.
// Every phase is parallel over tokens and channels, and the loads of a block are all in flight at once.
constexpr int kTileRowBytes = 256;

template <typename T>
__device__ __forceinline__ float2 ld2(const T* p);
template <>
__device__ __forceinline__ float2 ld2<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
template <>
__device__ __forceinline__ float2 ld2<float>(const float* p) {
    return *reinterpret_cast<const float2*>(p);
}

template <typename T, int K>
__global__ void __launch_bounds__(kThreads)
conv_bwd_tile_kernel(const T* __restrict__ x, long long xs, const float* __restrict__ w, const T* __restrict__ cache_in,
                     const T* __restrict__ dy, const T* __restrict__ dco, float* __restrict__ dx,
                     float* __restrict__ dcache, float* __restrict__ partial, const int32_t* __restrict__ cu, int nseq,
                     int T_len, int C) {
    constexpr int CB = kTileRowBytes / (int)sizeof(T);   // channels of the block
    constexpr int V16N = 16 / (int)sizeof(T);           // channels in 16 bytes
    constexpr int VPR = CB / V16N;                      // 16-byte vectors a row (16)
    constexpr int RX = kSlot + 2 * (K - 1), RD = kSlot + K - 1;
    constexpr int P = CB / 2, NG = kThreads / P;        // channel pairs; token groups
    extern __shared__ __align__(16) uint8_t smem[];
    T* sx = reinterpret_cast<T*>(smem);                                  // [RX][CB]
    T* sdy = sx + RX * CB;                                               // [RD][CB]
    float* sdu = reinterpret_cast<float*>(sdy + RD * CB);                // [RD][CB]
    const int tid = threadIdx.x;
    const int nblk = (C + CB - 1) / CB;
    const long long slot = blockIdx.x / nblk;
    const int cb0 = (int)(blockIdx.x % nblk) * CB;
    const int pr = tid % P, grp = tid / P, c = cb0 + 2 * pr;
    const bool cok = c < C;
    float* part = partial ? partial + ((size_t)slot * C + c) * K : nullptr;
    int seq, n;
    long long t0;
    if (!conv_slot(cu, nseq, T_len, slot, seq, t0, n)) {   // an unused slot adds nothing
        if (part && cok)
            for (int i = 0; i < 2 * K; ++i) part[i] = 0.f;
        return;
    }
    long long s0, s1;
    seq_range(cu, seq, T_len, s0, s1);
    // 1. rows to shared memory: every load of the thread issued before the first store
    // thread tid moves 16-byte piece q = tid % VPR of rows tid / VPR, + kThreads / VPR, ...
    constexpr int RPP = kThreads / VPR, NLD = (RX + RD + RPP - 1) / RPP;
    static_assert(kThreads % VPR == 0, "whole rows per pass");
    const int q = tid % VPR, rb = tid / VPR, cc = cb0 + q * V16N;
    const bool qok = cc < C;
    const int xlo = (int)(s0 - (t0 - (K - 1))), xhi = (int)min((long long)RX, s1 - (t0 - (K - 1)));   // x rows [xlo, xhi) are inputs
    const int dhi = (int)min((long long)RD, s1 - t0);                                                   // dy rows [0, dhi)
    // element offsets of row 0 (formed into pointers only for rows that exist): x row r is token
    // t0 - (K - 1) + r; before the sequence it is cache row r - xlo + K - 1 (only in a first slot, xlo > 0)
    const long long xoff0 = (t0 - (K - 1)) * xs + cc;
    const long long coff0 = ((long long)seq * (K - 1) + (K - 1) - xlo) * C + cc;
    const long long doff0 = t0 * (long long)C + cc;
    uint4 v[NLD];
#pragma unroll
    for (int k = 0; k < NLD; ++k) {
        const int r = rb + k * RPP;
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        if (qok && r < RX + RD) {
            if (r < RX) {
                if (r >= xlo && r < xhi)
                    v[k] = *reinterpret_cast<const uint4*>(x + (xoff0 + (long long)r * xs));
                else if (r < xlo && cache_in)
                    v[k] = *reinterpret_cast<const uint4*>(cache_in + (coff0 + (long long)r * C));
            } else if (r - RX < dhi) {
                v[k] = *reinterpret_cast<const uint4*>(dy + (doff0 + (long long)(r - RX) * C));
            }
        }
    }
#pragma unroll
    for (int k = 0; k < NLD; ++k) {
        const int r = rb + k * RPP;
        if (r < RX + RD) *reinterpret_cast<uint4*>((r < RX ? sx + r * CB : sdy + (r - RX) * CB) + q * V16N) = v[k];
    }
    float wv[2][K], acc[2][K];
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int j = 0; j < K; ++j) {
            wv[e][j] = cok ? w[(size_t)(c + e) * K + j] : 0.f;
            acc[e][j] = 0.f;
        }
    __syncthreads();
    // 2. du of the slot's tokens and the K - 1 after (zero past the sequence): each thread a channel pair
    //    and a run of consecutive tokens, the K x rows of a token sliding through registers
    constexpr int LR = (RD + NG - 1) / NG;          // tokens of a run
    const int nd = (int)min((long long)RD, s1 - t0);   // tokens with a du (the rest are past the sequence)
    {
        const int r0 = grp * LR;
        float2 xw[K];
#pragma unroll
        for (int j = 0; j + 1 < K; ++j) xw[j + 1] = ld2<T>(sx + (r0 + j) * CB + 2 * pr);
#pragma unroll
        for (int i = 0; i < LR; ++i) {
            const int r = r0 + i;
            if (r >= RD) break;
#pragma unroll
            for (int j = 0; j + 1 < K; ++j) xw[j] = xw[j + 1];
            xw[K - 1] = ld2<T>(sx + (r + K - 1) * CB + 2 * pr);
            float2 d = make_float2(0.f, 0.f);
            if (r < nd) {
                const float2 g = ld2<T>(sdy + r * CB + 2 * pr);
                float u0 = 0.f, u1 = 0.f;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    u0 = fmaf(wv[0][j], xw[j].x, u0);
                    u1 = fmaf(wv[1][j], xw[j].y, u1);
                }
                // sigmoid by the fast reciprocal; the clamp keeps 1 + e^-u finite and the result normal
                const float g0 = __fdividef(1.f, 1.f + __expf(fminf(-u0, 80.f)));
                const float g1 = __fdividef(1.f, 1.f + __expf(fminf(-u1, 80.f)));
                d = make_float2(g.x * g0 * (1.f + u0 * (1.f - g0)), g.y * g1 * (1.f + u1 * (1.f - g1)));
                if (r < n) {
#pragma unroll
                    for (int j = 0; j < K; ++j) {
                        acc[0][j] = fmaf(d.x, xw[j].x, acc[0][j]);
                        acc[1][j] = fmaf(d.y, xw[j].y, acc[1][j]);
                    }
                }
            }
            *reinterpret_cast<float2*>(sdu + r * CB + 2 * pr) = d;
        }
    }
    __syncthreads();
    // 3. dx of the slot's tokens, and of the cached inputs in a sequence's first slot: each thread a run of
    //    consecutive positions, the K du rows sliding through registers
    const int r_lo = (K > 1 && dcache && t0 == s0) ? -(K - 1) : 0;
    constexpr int LP = (kSlot + K - 1 + NG - 1) / NG;   // positions of a run (at most 64 + K - 1)
    // first position (relative to t0) that the outgoing cache holds; beyond any position of the slot if later
    const int dco_from = (int)min(s1 - (K - 1) - t0, (long long)kSlot);
    if (cok) {
        const int q0 = r_lo + grp * LP;
        float2 dw_[K];   // du rows q .. q + K - 1 (zero before the slot)
#pragma unroll
        for (int j = 0; j + 1 < K; ++j) {
            const int rd = q0 + j;
            dw_[j + 1] = rd >= 0 ? *reinterpret_cast<const float2*>(sdu + rd * CB + 2 * pr) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < LP; ++i) {
            const int r = q0 + i;
            if (r >= n) break;
#pragma unroll
            for (int j = 0; j + 1 < K; ++j) dw_[j] = dw_[j + 1];
            const int rd = r + K - 1;
            dw_[K - 1] = rd >= 0 ? *reinterpret_cast<const float2*>(sdu + rd * CB + 2 * pr) : make_float2(0.f, 0.f);
            float2 gx = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < K; ++j) {   // du of token p + K - 1 - j is dw_[K - 1 - j]
                gx.x = fmaf(wv[0][j], dw_[K - 1 - j].x, gx.x);
                gx.y = fmaf(wv[1][j], dw_[K - 1 - j].y, gx.y);
            }
            const long long p = t0 + r;
            if (dco && r >= dco_from) {   // the outgoing cache holds this input
                const float2 gc = ld2<T>(dco + ((size_t)seq * (K - 1) + (size_t)(r - dco_from)) * C + c);
                gx.x += gc.x;
                gx.y += gc.y;
            }
            float* dst = r >= 0 ? dx + p * (long long)C + c
                                : dcache + ((size_t)seq * (K - 1) + (size_t)(r + K - 1)) * C + c;
            *reinterpret_cast<float2*>(dst) = gx;
        }
    }
    // 4. the token groups' tap sums, added in group order
    __syncthreads();
    float* red = reinterpret_cast<float*>(smem);   // [NG][P][2K] over the staged rows
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int j = 0; j < K; ++j) red[(grp * P + pr) * 2 * K + e * K + j] = acc[e][j];
    __syncthreads();
    if (part && grp == 0 && cok) {
#pragma unroll
        for (int i = 0; i < 2 * K; ++i) {
            float t = 0.f;
            for (int g = 0; g < NG; ++g) t += red[(g * P + pr) * 2 * K + i];
            part[i] = t;   // channel c + i / K, tap i % K: [c][K] then [c + 1][K]
        }
    }
}

template <typename T, int K>
constexpr size_t tile_smem_bytes() {
    constexpr int CB = kTileRowBytes / (int)sizeof(T);
    return (size_t)(kSlot + 2 * (K - 1)) * kTileRowBytes + (size_t)(kSlot + K - 1) * kTileRowBytes +
           (size_t)(kSlot + K - 1) * CB * sizeof(float);
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
    const long long slots = conv_slots(a);
    const int T_len = a.T;
    const int32_t* cu = a.packed ? a.cu_seqlens : nullptr;
    constexpr size_t smem = tile_smem_bytes<T, K>();
    const long long blocks = slots * ((a.C + kTileRowBytes / (int)sizeof(T) - 1) / (kTileRowBytes / (int)sizeof(T)));
    if (blocks > 0) {
        cudaError_t e = cudaFuncSetAttribute(conv_bwd_tile_kernel<T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        conv_bwd_tile_kernel<T, K><<<(unsigned)blocks, kThreads, smem, a.stream>>>(
            static_cast<const T*>(a.x), a.x_stride, a.w, static_cast<const T*>(a.cache_in), static_cast<const T*>(dy),
            static_cast<const T*>(dco), dx, dcache, partial, cu, a.num_seqs, T_len, a.C);
    }
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
