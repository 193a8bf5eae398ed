// Recurrent decode step (one new token per sequence), memory-bound.
//
// Per (sequence n, value head h), with a = exp(g), state S (dk x dv, fp32), query/key head
// h / (Hv/Hqk), the step of "Transformer by Hand, ch. 7", section "The formula":
//     p = S^T k,  r = S^T q            (both from the state before the decay; one read)
//     u = beta (v - a p)               (the delta written for this token)
//     S <- a S + k u^T                 (one write)
//     o = scale (a r + (k . q) u)      (= scale S_new^T q, expanded so the state is read once)
// With GDN_RAW_GATES, g and beta hold the raw projections and the gates are formed here; with
// GDN_OUTPUT_GATE the outputs pass through the shell's gated RMS normalisation before they are stored.
//
// One CTA of 256 threads owns one (n, h) table.  Thread (row group rg, column lane lx) holds
// rows rg*RPT .. rg*RPT+RPT-1 and four adjacent columns 4*lx .. 4*lx+3 in registers; the loads
// and stores are 128-bit and a warp covers whole contiguous rows (fully coalesced).  The two
// column reductions over dk go through shared memory once.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecThreads = 256;

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kDecThreads, 2)
decode_step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ g, const T* __restrict__ beta, float* __restrict__ S,
                   T* __restrict__ out, int Hqk, int Hv, float scale, int normalize,
                   const float* __restrict__ A_log, const float* __restrict__ dt_bias,
                   const T* __restrict__ zg, const float* __restrict__ norm_w, float norm_eps) {
    constexpr int LX = DV / 4;                 // column lanes (float4 each)
    constexpr int RG = kDecThreads / LX;       // row groups
    constexpr int RPT = DK / RG;               // rows per thread
    static_assert(RPT >= 1 && DK % RG == 0, "tile");

    __shared__ __align__(16) float sk[DK];
    __shared__ __align__(16) float sq[DK];
    __shared__ __align__(16) float sv[DV];
    __shared__ __align__(16) float su[DV];
    __shared__ __align__(16) float red_p[RG][DV + 4];   // rows of DV+4 floats stay 16-byte aligned
    __shared__ __align__(16) float red_r[RG][DV + 4];
    __shared__ __align__(16) float so[DV];   // outputs kept for the output gate
    __shared__ float s_kq, s_rk, s_rq, s_inv;

    const int nh = blockIdx.x;                 // n * Hv + h
    const int n = nh / Hv, h = nh % Hv;
    const int hk = h / (Hv / Hqk);
    const int tid = threadIdx.x;
    const int lx = tid % LX, rg = tid / LX;

    float4* Sv = reinterpret_cast<float4*>(S + (size_t)nh * DK * DV);
    float4 st[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) st[r] = Sv[(size_t)(rg * RPT + r) * LX + lx];

    const T* qp = q + ((size_t)n * Hqk + hk) * DK;
    const T* kp = k + ((size_t)n * Hqk + hk) * DK;
    for (int i = tid; i < DK; i += kDecThreads) {
        sq[i] = to_f32(qp[i]);
        sk[i] = to_f32(kp[i]);
    }
    for (int j = tid; j < DV; j += kDecThreads) sv[j] = to_f32(v[(size_t)nh * DV + j]);
    float gt = to_f32(g[nh]), bt = to_f32(beta[nh]);
    if (A_log) gates_from_raw(gt, bt, A_log[h], dt_bias[h], gt, bt);   // raw projections a, b
    const float alpha = __expf(gt);
    __syncthreads();

    if (tid < 32) {                            // k.q and, if asked, the norms of k and q
        float kq = 0.f, kk = 0.f, qq = 0.f;
        for (int i = tid; i < DK; i += 32) {
            kq = fmaf(sk[i], sq[i], kq);
            kk = fmaf(sk[i], sk[i], kk);
            qq = fmaf(sq[i], sq[i], qq);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            kq += __shfl_xor_sync(0xffffffffu, kq, o);
            kk += __shfl_xor_sync(0xffffffffu, kk, o);
            qq += __shfl_xor_sync(0xffffffffu, qq, o);
        }
        if (tid == 0) {
            const float rk = normalize ? rsqrtf(kk + 1e-6f) : 1.f;
            const float rq = normalize ? rsqrtf(qq + 1e-6f) : 1.f;
            s_kq = kq * rk * rq;
            s_rk = rk;
            s_rq = rq;
        }
    }
    __syncthreads();
    const float rk = s_rk, rq = s_rq;

    float p[4] = {0.f, 0.f, 0.f, 0.f}, rr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const float kr = sk[rg * RPT + r], qr = sq[rg * RPT + r];
        p[0] = fmaf(st[r].x, kr, p[0]); p[1] = fmaf(st[r].y, kr, p[1]);
        p[2] = fmaf(st[r].z, kr, p[2]); p[3] = fmaf(st[r].w, kr, p[3]);
        rr[0] = fmaf(st[r].x, qr, rr[0]); rr[1] = fmaf(st[r].y, qr, rr[1]);
        rr[2] = fmaf(st[r].z, qr, rr[2]); rr[3] = fmaf(st[r].w, qr, rr[3]);
    }
    reinterpret_cast<float4*>(&red_p[rg][0])[lx] = make_float4(p[0], p[1], p[2], p[3]);
    reinterpret_cast<float4*>(&red_r[rg][0])[lx] = make_float4(rr[0], rr[1], rr[2], rr[3]);
    __syncthreads();

    if (tid < DV) {
        float pj = 0.f, rj = 0.f;
#pragma unroll 8
        for (int x = 0; x < RG; ++x) {
            pj += red_p[x][tid];
            rj += red_r[x][tid];
        }
        pj *= rk;                                // S^T k_hat
        rj *= rq;                                // S^T q_hat
        const float u = bt * (sv[tid] - alpha * pj);
        su[tid] = u;
        const float o = scale * fmaf(alpha, rj, s_kq * u);
        if (zg) so[tid] = o;
        else out[(size_t)nh * DV + tid] = from_f32<T>(o);
    }
    __syncthreads();

    const float4 uu = reinterpret_cast<const float4*>(su)[lx];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const float kr = sk[rg * RPT + r] * rk;
        float4 o;
        o.x = fmaf(kr, uu.x, alpha * st[r].x);
        o.y = fmaf(kr, uu.y, alpha * st[r].y);
        o.z = fmaf(kr, uu.z, alpha * st[r].z);
        o.w = fmaf(kr, uu.w, alpha * st[r].w);
        Sv[(size_t)(rg * RPT + r) * LX + lx] = o;
    }
    if (zg) {   // output gate: o / sqrt(mean(o^2) + eps) * w * silu(z), after the state is written
        __syncthreads();
        if (tid < 32) {
            float ss = 0.f;
            for (int j = tid; j < DV; j += 32) ss = fmaf(so[j], so[j], ss);
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            if (tid == 0) s_inv = rsqrtf(ss / (float)DV + norm_eps);
        }
        __syncthreads();
        if (tid < DV)
            out[(size_t)nh * DV + tid] =
                from_f32<T>(so[tid] * s_inv * norm_w[tid] * silu_for<T>(to_f32(zg[(size_t)nh * DV + tid])));
    }
}

template <int DK, int DV, typename T>
cudaError_t launch_typed(const DecodeArgs& a) {
    const unsigned blocks = (unsigned)((long long)a.N * a.Hv);
    decode_step_kernel<DK, DV, T><<<blocks, kDecThreads, 0, a.stream>>>(
        static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
        static_cast<const T*>(a.g), static_cast<const T*>(a.beta), a.S, static_cast<T*>(a.out), a.Hqk,
        a.Hv, a.scale, (a.flags & GDN_NORMALIZE_QK) ? 1 : 0, (a.flags & GDN_RAW_GATES) ? a.A_log : nullptr,
        a.dt_bias, (a.flags & GDN_OUTPUT_GATE) ? static_cast<const T*>(a.z) : nullptr, a.norm_weight, a.norm_eps);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dims(const DecodeArgs& a) {
#define GDN_DEC_CASE(DK_, DV_) \
    if (a.dk == DK_ && a.dv == DV_) return launch_typed<DK_, DV_, T>(a);
    GDN_DEC_CASE(32, 32) GDN_DEC_CASE(32, 64) GDN_DEC_CASE(32, 128)
    GDN_DEC_CASE(64, 32) GDN_DEC_CASE(64, 64) GDN_DEC_CASE(64, 128)
    GDN_DEC_CASE(128, 32) GDN_DEC_CASE(128, 64) GDN_DEC_CASE(128, 128)
#undef GDN_DEC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a) {
    if (a.N == 0) return cudaSuccess;
    return a.dtype == GDN_BF16 ? launch_dims<__nv_bfloat16>(a) : launch_dims<float>(a);
}

}  // namespace gdn
