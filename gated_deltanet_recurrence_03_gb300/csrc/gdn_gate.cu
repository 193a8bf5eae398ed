// Output gate of the GatedDeltaNet shell ("Transformer by Hand, ch. 7", listing "qwen/deltanet.py":
// out = self.norm(out, z) with GatedRMSNorm, and the parts table: "the output is normalised per head
// and then multiplied by the gate silu(z)"):
//     y_j = o_j / sqrt(mean_j(o_j^2) + eps) * w_j * silu(z_j)      over the dv values of one (token, head)
// A memory-bound pass (16-byte vectors, a lane group per row), in place over `out` after the prefill
// kernels, whose outputs are split across CTAs by value columns, or from o to y for the standalone entry
// point.  The decode kernel applies the same gate in its own epilogue.  The backward below gives the
// gradients with respect to o, z and the weight.
#include <algorithm>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerThread = 2;   // independent rows per thread, for loads in flight

// 16-byte vectors: a group of DV / VEC lanes holds one row; a warp holds 32 / (DV / VEC) rows per pass.
template <typename T>
struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
    __device__ static void load(const T* p, float* f) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int e = 0; e < N; ++e) f[e] = to_f32(h[e]);
    }
    __device__ static void store(T* p, const float* f) {
        uint4 u;
        T* h = reinterpret_cast<T*>(&u);
#pragma unroll
        for (int e = 0; e < N; ++e) h[e] = from_f32<T>(f[e]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};

template <int DV, typename T>
__global__ void __launch_bounds__(32 * kWarps)
output_gate_kernel(const T* in, T* out, const T* __restrict__ z, const float* __restrict__ w, float eps,
                   long long rows) {
    constexpr int VEC = Vec16<T>::N;
    constexpr int LPR = DV / VEC;          // lanes per row
    constexpr int RPW = 32 / LPR;          // rows per warp and pass
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row must split evenly over a warp");
    const int lane = threadIdx.x & 31, sub = lane % LPR;
    const long long warp = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    float wv[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) wv[e] = w[sub * VEC + e];
    long long row[kRowsPerThread];
    float o[kRowsPerThread][VEC], zz[kRowsPerThread][VEC], ss[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        row[r] = (warp * kRowsPerThread + r) * RPW + lane / LPR;
        ss[r] = 0.f;
        if (row[r] < rows) {
            Vec16<T>::load(in + row[r] * DV + sub * VEC, o[r]);
            Vec16<T>::load(z + row[r] * DV + sub * VEC, zz[r]);
#pragma unroll
            for (int e = 0; e < VEC; ++e) ss[r] = fmaf(o[r][e], o[r][e], ss[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
#pragma unroll
        for (int m = LPR / 2; m > 0; m >>= 1) ss[r] += __shfl_xor_sync(0xffffffffu, ss[r], m);
        if (row[r] >= rows) continue;
        const float inv = rsqrtf(ss[r] / (float)DV + eps);
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[r][e] = o[r][e] * inv * wv[e] * silu_for<T>(zz[r][e]);
        Vec16<T>::store(out + row[r] * DV + sub * VEC, o[r]);
    }
}

template <int DV, typename T>
cudaError_t launch_dv(const void* in, void* out, const void* z, const float* w, float eps, long long rows,
                      cudaStream_t stream) {
    constexpr int RPW = 32 / (DV / Vec16<T>::N);
    const long long per_block = (long long)kWarps * kRowsPerThread * RPW;
    const unsigned blocks = (unsigned)((rows + per_block - 1) / per_block);
    output_gate_kernel<DV, T><<<blocks, 32 * kWarps, 0, stream>>>(static_cast<const T*>(in), static_cast<T*>(out),
                                                                  static_cast<const T*>(z), w, eps, rows);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const void* in, void* out, const void* z, const float* w, float eps, long long rows, int dv,
                         cudaStream_t stream) {
    switch (dv) {
        case 32: return launch_dv<32, T>(in, out, z, w, eps, rows, stream);
        case 64: return launch_dv<64, T>(in, out, z, w, eps, rows, stream);
        case 128: return launch_dv<128, T>(in, out, z, w, eps, rows, stream);
    }
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- backward
// With inv = (mean(o^2) + eps)^-1/2, o_hat = o inv, s = silu(z) and gy = dy w s, per row:
//     do = inv (gy - o_hat mean(gy o_hat)),   dz = dy o_hat w silu'(z),
// and dw = sum over the rows of dy o_hat s: each block sums its rows' terms per column (threads of a
// column in a fixed order) into partial[block][dv]; column_sum_kernel adds the blocks in a fixed order.
constexpr int kBwdBlocksMax = 1024;

// Four values per lane (8 bytes of bf16, 16 of fp32): a warp holds 32 / (DV / 4) rows per pass, the state
// of a thread stays small, and the next pass's raw o, z, dy are loaded while this pass computes.
template <typename T>
struct Vec8;
template <>
struct Vec8<__nv_bfloat16> {
    static constexpr int N = 4;
    using Raw = uint2;
    __device__ static void unpack(const Raw& u, float* f) {
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
        for (int e = 0; e < N; ++e) f[e] = __bfloat162float(h[e]);
    }
};
template <>
struct Vec8<float> {
    static constexpr int N = 4;
    using Raw = uint4;
    __device__ static void unpack(const Raw& u, float* f) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
};

template <int N>
__device__ __forceinline__ void store_f32(float* p, const float (&f)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int e = 0; e < N; e += 4) *reinterpret_cast<float4*>(p + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
    } else {
        static_assert(N == 2, "two or a multiple of four values");
        *reinterpret_cast<float2*>(p) = make_float2(f[0], f[1]);
    }
}

template <int DV, typename T>
__global__ void __launch_bounds__(32 * kWarps)
output_gate_bwd_kernel(const T* __restrict__ o_in, const T* __restrict__ z, const float* __restrict__ w, float eps,
                       const T* __restrict__ dy_in, float* __restrict__ d_o, float* __restrict__ d_z,
                       float* __restrict__ partial, long long rows) {
    constexpr int VEC = Vec8<T>::N;
    constexpr int LPR = DV / VEC;          // lanes per row
    constexpr int RPW = 32 / LPR;          // rows per warp and pass
    constexpr int THREADS = 32 * kWarps;
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row must split evenly over a warp");
    __shared__ float red[THREADS][VEC + 1];
    const int tid = threadIdx.x, lane = tid & 31, sub = lane % LPR;
    float wv[VEC], acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        wv[e] = w[sub * VEC + e];
        acc[e] = 0.f;
    }
    const long long rows_per_pass = (long long)gridDim.x * kWarps * RPW;
    long long row = ((long long)blockIdx.x * kWarps + (tid >> 5)) * RPW + lane / LPR;
    using Raw = typename Vec8<T>::Raw;
    const auto fetch = [&](long long r, Raw& ro, Raw& rz, Raw& rd) {
        if (r < rows) {
            const size_t off = (size_t)r * DV + sub * VEC;
            ro = *reinterpret_cast<const Raw*>(o_in + off);
            rz = *reinterpret_cast<const Raw*>(z + off);
            rd = *reinterpret_cast<const Raw*>(dy_in + off);
        }
    };
    Raw no{}, nz{}, nd{};
    fetch(row, no, nz, nd);
    for (; row - lane / LPR < rows; row += rows_per_pass) {   // warp-uniform: the warp's first row
        const bool ok = row < rows;
        float o[VEC], zz[VEC], dy[VEC];
        Vec8<T>::unpack(no, o);
        Vec8<T>::unpack(nz, zz);
        Vec8<T>::unpack(nd, dy);
        fetch(row + rows_per_pass, no, nz, nd);   // the next pass's rows, while this one computes
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) ss = fmaf(o[e], o[e], ss);
#pragma unroll
        for (int m = LPR / 2; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float inv = rsqrtf(ss / (float)DV + eps);
        float gy[VEC], sg[VEC], dot = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            // sigmoid by the fast reciprocal; the clamp keeps 1 + e^-z finite and the result normal
            sg[e] = __fdividef(1.f, 1.f + __expf(fminf(-zz[e], 80.f)));
            gy[e] = dy[e] * wv[e] * zz[e] * sg[e];
            dot = fmaf(gy[e], o[e] * inv, dot);
        }
#pragma unroll
        for (int m = LPR / 2; m > 0; m >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
        if (!ok) continue;
        const float mdot = dot / (float)DV;
        float rdo[VEC], rdz[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float sig = sg[e], oh = o[e] * inv;
            rdo[e] = inv * (gy[e] - oh * mdot);
            rdz[e] = dy[e] * oh * wv[e] * sig * (1.f + zz[e] * (1.f - sig));
            acc[e] = fmaf(dy[e] * oh, zz[e] * sig, acc[e]);
        }
        store_f32(d_o + row * DV + sub * VEC, rdo);
        store_f32(d_z + row * DV + sub * VEC, rdz);
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) red[tid][e] = acc[e];
    __syncthreads();
    // column c = sub * VEC + e is held by every thread whose lane % LPR == sub: add them in thread order
    for (int c = tid; c < DV; c += THREADS) {
        const int sb = c / VEC, e = c % VEC;
        float t = 0.f;
        for (int th = sb; th < THREADS; th += LPR) t += red[th][e];
        partial[(size_t)blockIdx.x * DV + c] = t;
    }
}

template <int DV, typename T>
int bwd_blocks(long long rows) {
    constexpr int RPW = 32 / (DV / Vec8<T>::N);
    const long long per_block = (long long)kWarps * RPW;
    return (int)std::min<long long>(std::max<long long>((rows + per_block - 1) / per_block, 1), kBwdBlocksMax);
}

template <int DV, typename T>
cudaError_t launch_bwd_dv(const void* o, const void* z, const float* w, float eps, const void* dy, float* d_o,
                          float* d_z, float* d_w, float* partial, long long rows, cudaStream_t stream) {
    const int blocks = bwd_blocks<DV, T>(rows);
    output_gate_bwd_kernel<DV, T><<<blocks, 32 * kWarps, 0, stream>>>(
        static_cast<const T*>(o), static_cast<const T*>(z), w, eps, static_cast<const T*>(dy), d_o, d_z, partial, rows);
    if (d_w) column_sum_kernel<<<(DV + 31) / 32, kColSumThreads, 0, stream>>>(partial, blocks, DV, d_w);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_typed(const void* o, const void* z, const float* w, float eps, const void* dy, float* d_o,
                             float* d_z, float* d_w, float* partial, long long rows, int dv, cudaStream_t stream) {
    switch (dv) {
        case 32: return launch_bwd_dv<32, T>(o, z, w, eps, dy, d_o, d_z, d_w, partial, rows, stream);
        case 64: return launch_bwd_dv<64, T>(o, z, w, eps, dy, d_o, d_z, d_w, partial, rows, stream);
        case 128: return launch_bwd_dv<128, T>(o, z, w, eps, dy, d_o, d_z, d_w, partial, rows, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_output_gate(void* out, const void* z, const float* w, float eps, long long rows, int dv,
                               int dtype, cudaStream_t stream) {
    return launch_output_gate_to(out, out, z, w, eps, rows, dv, dtype, stream);
}

cudaError_t launch_output_gate_to(const void* in, void* out, const void* z, const float* w, float eps, long long rows,
                                  int dv, int dtype, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    return dtype == GDN_BF16 ? launch_typed<__nv_bfloat16>(in, out, z, w, eps, rows, dv, stream)
                             : launch_typed<float>(in, out, z, w, eps, rows, dv, stream);
}

__global__ void __launch_bounds__(kColSumThreads)
column_sum_kernel(const float* __restrict__ in, long long rows, int cols, float* __restrict__ out) {
    __shared__ float red[32][33];
    const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5, c = blockIdx.x * 32 + lane;
    float t = 0.f;
    if (c < cols) {
#pragma unroll 4
        for (long long r = grp; r < rows; r += 32) t += in[(size_t)r * cols + c];
    }
    red[grp][lane] = t;
    __syncthreads();
    for (int w = 16; w > 0; w >>= 1) {
        if (grp < w) red[grp][lane] += red[grp + w][lane];
        __syncthreads();
    }
    if (grp == 0 && c < cols) out[c] = red[0][lane];
}

size_t output_gate_bwd_workspace_bytes(long long rows, int dv) {
    (void)rows;
    return (size_t)kBwdBlocksMax * dv * sizeof(float);
}

cudaError_t launch_output_gate_bwd(const void* o, const void* z, const float* w, float eps, const void* dy, float* d_o,
                                   float* d_z, float* d_w, void* workspace, long long rows, int dv, int dtype,
                                   cudaStream_t stream) {
    float* partial = static_cast<float*>(workspace);
    if (rows <= 0) {   // no rows: the weight gradient is zero
        if (d_w) {
            const cudaError_t e = cudaMemsetAsync(d_w, 0, (size_t)dv * sizeof(float), stream);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    return dtype == GDN_BF16 ? launch_bwd_typed<__nv_bfloat16>(o, z, w, eps, dy, d_o, d_z, d_w, partial, rows, dv, stream)
                             : launch_bwd_typed<float>(o, z, w, eps, dy, d_o, d_z, d_w, partial, rows, dv, stream);
}

}  // namespace gdn
