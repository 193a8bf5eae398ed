// Output gate of the GatedDeltaNet shell ("Transformer by Hand, ch. 7", listing "qwen/deltanet.py":
// out = self.norm(out, z) with GatedRMSNorm, and the parts table: "the output is normalised per head
// and then multiplied by the gate silu(z)"):
//     y_j = o_j / sqrt(mean_j(o_j^2) + eps) * w_j * silu(z_j)      over the dv values of one (token, head)
// A memory-bound pass over `out` in place (one warp per row), used after the prefill kernels, whose
// outputs are split across CTAs by value columns.  The decode kernel applies the same gate in its
// own epilogue.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRowsPerBlock = 8;

template <int DV, typename T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
output_gate_kernel(T* __restrict__ out, const T* __restrict__ z, const float* __restrict__ w, float eps,
                   long long rows) {
    constexpr int PER = DV / 32;
    const long long row = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    T* orow = out + row * DV + lane * PER;
    const T* zrow = z + row * DV + lane * PER;
    float o[PER], zz[PER];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        o[e] = to_f32(orow[e]);
        zz[e] = to_f32(zrow[e]);
        ss = fmaf(o[e], o[e], ss);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float inv = rsqrtf(ss / (float)DV + eps);
#pragma unroll
    for (int e = 0; e < PER; ++e) orow[e] = from_f32<T>(o[e] * inv * w[lane * PER + e] * silu_f(zz[e]));
}

template <typename T>
cudaError_t launch_typed(void* out, const void* z, const float* w, float eps, long long rows, int dv,
                         cudaStream_t stream) {
    const unsigned blocks = (unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    if (dv == 32)
        output_gate_kernel<32, T><<<blocks, 32 * kRowsPerBlock, 0, stream>>>(static_cast<T*>(out), static_cast<const T*>(z), w, eps, rows);
    else if (dv == 64)
        output_gate_kernel<64, T><<<blocks, 32 * kRowsPerBlock, 0, stream>>>(static_cast<T*>(out), static_cast<const T*>(z), w, eps, rows);
    else if (dv == 128)
        output_gate_kernel<128, T><<<blocks, 32 * kRowsPerBlock, 0, stream>>>(static_cast<T*>(out), static_cast<const T*>(z), w, eps, rows);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_output_gate(void* out, const void* z, const float* w, float eps, long long rows, int dv,
                               int dtype, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    return dtype == GDN_BF16 ? launch_typed<__nv_bfloat16>(out, z, w, eps, rows, dv, stream)
                             : launch_typed<float>(out, z, w, eps, rows, dv, stream);
}

}  // namespace gdn
