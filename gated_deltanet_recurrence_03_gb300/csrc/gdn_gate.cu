// Output gate of the GatedDeltaNet shell ("Transformer by Hand, ch. 7", listing "qwen/deltanet.py":
// out = self.norm(out, z) with GatedRMSNorm, and the parts table: "the output is normalised per head
// and then multiplied by the gate silu(z)"):
//     y_j = o_j / sqrt(mean_j(o_j^2) + eps) * w_j * silu(z_j)      over the dv values of one (token, head)
// A memory-bound pass over `out` in place (16-byte vectors, a lane group per row), used after the prefill kernels, whose
// outputs are split across CTAs by value columns.  The decode kernel applies the same gate in its
// own epilogue.
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
output_gate_kernel(T* __restrict__ out, const T* __restrict__ z, const float* __restrict__ w, float eps,
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
            Vec16<T>::load(out + row[r] * DV + sub * VEC, o[r]);
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
cudaError_t launch_dv(void* out, const void* z, const float* w, float eps, long long rows, cudaStream_t stream) {
    constexpr int RPW = 32 / (DV / Vec16<T>::N);
    const long long per_block = (long long)kWarps * kRowsPerThread * RPW;
    const unsigned blocks = (unsigned)((rows + per_block - 1) / per_block);
    output_gate_kernel<DV, T><<<blocks, 32 * kWarps, 0, stream>>>(static_cast<T*>(out), static_cast<const T*>(z), w,
                                                                  eps, rows);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(void* out, const void* z, const float* w, float eps, long long rows, int dv,
                         cudaStream_t stream) {
    switch (dv) {
        case 32: return launch_dv<32, T>(out, z, w, eps, rows, stream);
        case 64: return launch_dv<64, T>(out, z, w, eps, rows, stream);
        case 128: return launch_dv<128, T>(out, z, w, eps, rows, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_output_gate(void* out, const void* z, const float* w, float eps, long long rows, int dv,
                               int dtype, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    return dtype == GDN_BF16 ? launch_typed<__nv_bfloat16>(out, z, w, eps, rows, dv, stream)
                             : launch_typed<float>(out, z, w, eps, rows, dv, stream);
}

}  // namespace gdn
