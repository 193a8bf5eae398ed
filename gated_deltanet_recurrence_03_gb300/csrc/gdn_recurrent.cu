// Token-serial prefill on CUDA cores: the recurrence of "Transformer by Hand, ch. 7" (section
// "The formula"; the four steps of the delta_rule listing) run token by token in fp32.
//
// It serves fp32 inputs (whose 1e-4 parity budget rules out bf16/tf32 tensor-core operands) and
// the head shapes the tensor-core chunked kernel does not take.  One CTA owns one
// (sequence, value head) table; dk/32 adjacent lanes own column j of S (32 rows each, in
// registers), so the lookups S^T k and S^T q are per-thread dot products combined by at most two
// warp shuffles, with no shared-memory reduction inside the token loop.  Inputs are staged
// through shared memory TB tokens at a time; k.q and the optional l2 normalisation are computed
// while staging.
//
//   per token:  p = S^T k,  r = S^T q  (state before the decay)
//               u = beta (v - a p),  S <- a S + k u^T,  o = scale (a r + (k.q) u)
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kTB = 16;  // tokens staged per round

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(DV * (DK / 32))
recurrent_prefill_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                         const T* __restrict__ g, const T* __restrict__ beta,
                         const float* __restrict__ S0, T* __restrict__ out, float* __restrict__ S_final,
                         const int32_t* __restrict__ cu, int T_len, int Hqk, int Hv, float scale,
                         int normalize, const float* __restrict__ A_log, const float* __restrict__ dt_bias) {
    constexpr int SPLIT = DK / 32;           // adjacent lanes sharing one column, 32 rows each
    constexpr int NT = DV * SPLIT;           // threads
    constexpr int NW = NT / 32;
    __shared__ __align__(16) float sk[kTB][DK];
    __shared__ __align__(16) float sq[kTB][DK];
    __shared__ float sv[kTB][DV];
    __shared__ float sa[kTB], sb[kTB], skq[kTB];

    const int h = blockIdx.x % Hv;
    const int i = blockIdx.x / Hv;
    const int hk = h / (Hv / Hqk);
    const int tid = threadIdx.x;
    const int j = tid / SPLIT;              // column of S
    const int part = tid % SPLIT;           // rows part*32 .. part*32+31
    const int lane = tid & 31, warp = tid >> 5;

    long long t0, t1;
    seq_range(cu, i, T_len, t0, t1);

    const size_t sbase = ((size_t)i * Hv + h) * DK * DV;
    float s[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) s[r] = S0 ? S0[sbase + (size_t)(part * 32 + r) * DV + j] : 0.f;

    for (long long tb = t0; tb < t1; tb += kTB) {
        const int nt = (int)min((long long)kTB, t1 - tb);
        __syncthreads();  // previous round finished with the staging buffers
        for (int e = tid; e < nt * DK; e += NT) {
            const int tt = e / DK, c = e % DK;
            const size_t off = ((size_t)(tb + tt) * Hqk + hk) * DK + c;
            sk[tt][c] = to_f32(k[off]);
            sq[tt][c] = to_f32(q[off]);
        }
        for (int e = tid; e < nt * DV; e += NT) {
            const int tt = e / DV, c = e % DV;
            sv[tt][c] = to_f32(v[((size_t)(tb + tt) * Hv + h) * DV + c]);
        }
        if (tid < nt) {
            float gt = to_f32(g[(size_t)(tb + tid) * Hv + h]), bt = to_f32(beta[(size_t)(tb + tid) * Hv + h]);
            if (A_log) gates_from_raw(gt, bt, A_log[h], dt_bias[h], gt, bt);   // raw projections a, b
            sa[tid] = __expf(gt);
            sb[tid] = bt;
        }
        __syncthreads();
        for (int tt = warp; tt < nt; tt += NW) {   // one warp per token: norms and k.q
            float kk = 0.f, qq = 0.f, kq = 0.f;
            for (int c = lane; c < DK; c += 32) {
                kk = fmaf(sk[tt][c], sk[tt][c], kk);
                qq = fmaf(sq[tt][c], sq[tt][c], qq);
                kq = fmaf(sk[tt][c], sq[tt][c], kq);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                kk += __shfl_xor_sync(0xffffffffu, kk, o);
                qq += __shfl_xor_sync(0xffffffffu, qq, o);
                kq += __shfl_xor_sync(0xffffffffu, kq, o);
            }
            if (normalize) {
                const float rk = rsqrtf(kk + 1e-6f), rq = rsqrtf(qq + 1e-6f);
                for (int c = lane; c < DK; c += 32) {
                    sk[tt][c] *= rk;
                    sq[tt][c] *= rq;
                }
                kq *= rk * rq;
            }
            if (lane == 0) skq[tt] = kq;
        }
        __syncthreads();

        for (int tt = 0; tt < nt; ++tt) {
            const float4* k4 = reinterpret_cast<const float4*>(sk[tt] + part * 32);
            const float4* q4 = reinterpret_cast<const float4*>(sq[tt] + part * 32);
            float p0 = 0.f, p1 = 0.f, r0 = 0.f, r1 = 0.f;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float4 kr = k4[r], qr = q4[r];
                p0 = fmaf(s[4 * r + 0], kr.x, p0); r0 = fmaf(s[4 * r + 0], qr.x, r0);
                p1 = fmaf(s[4 * r + 1], kr.y, p1); r1 = fmaf(s[4 * r + 1], qr.y, r1);
                p0 = fmaf(s[4 * r + 2], kr.z, p0); r0 = fmaf(s[4 * r + 2], qr.z, r0);
                p1 = fmaf(s[4 * r + 3], kr.w, p1); r1 = fmaf(s[4 * r + 3], qr.w, r1);
            }
            float p = p0 + p1, rr = r0 + r1;
#pragma unroll
            for (int o = 1; o < SPLIT; o <<= 1) {
                p += __shfl_xor_sync(0xffffffffu, p, o);
                rr += __shfl_xor_sync(0xffffffffu, rr, o);
            }
            const float a = sa[tt];
            const float u = sb[tt] * (sv[tt][j] - a * p);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float4 kr = k4[r];
                s[4 * r + 0] = fmaf(kr.x, u, a * s[4 * r + 0]);
                s[4 * r + 1] = fmaf(kr.y, u, a * s[4 * r + 1]);
                s[4 * r + 2] = fmaf(kr.z, u, a * s[4 * r + 2]);
                s[4 * r + 3] = fmaf(kr.w, u, a * s[4 * r + 3]);
            }
            if (part == 0)
                out[((size_t)(tb + tt) * Hv + h) * DV + j] = from_f32<T>(scale * fmaf(a, rr, skq[tt] * u));
        }
    }
    if (S_final) {
#pragma unroll
        for (int r = 0; r < 32; ++r) S_final[sbase + (size_t)(part * 32 + r) * DV + j] = s[r];
    }
}

template <int DK, int DV, typename T>
cudaError_t launch_typed(const PrefillArgs& a) {
    const unsigned blocks = (unsigned)((long long)a.num_seqs * a.Hv);
    const int T_len = a.T;
    recurrent_prefill_kernel<DK, DV, T><<<blocks, DV * (DK / 32), 0, a.stream>>>(
        static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
        static_cast<const T*>(a.g), static_cast<const T*>(a.beta), a.S0, static_cast<T*>(a.out),
        a.S_final, a.cu_seqlens, T_len, a.Hqk, a.Hv, a.scale, (a.flags & GDN_NORMALIZE_QK) ? 1 : 0,
        (a.flags & GDN_RAW_GATES) ? a.A_log : nullptr, a.dt_bias);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dims(const PrefillArgs& a) {
#define GDN_REC_CASE(DK_, DV_) \
    if (a.dk == DK_ && a.dv == DV_) return launch_typed<DK_, DV_, T>(a);
    GDN_REC_CASE(32, 32) GDN_REC_CASE(32, 64) GDN_REC_CASE(32, 128)
    GDN_REC_CASE(64, 32) GDN_REC_CASE(64, 64) GDN_REC_CASE(64, 128)
    GDN_REC_CASE(128, 32) GDN_REC_CASE(128, 64) GDN_REC_CASE(128, 128)
#undef GDN_REC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_recurrent_prefill(const PrefillArgs& a) {
    if (a.num_seqs == 0 || a.Hv == 0) return cudaSuccess;
    return a.dtype == GDN_BF16 ? launch_dims<__nv_bfloat16>(a) : launch_dims<float>(a);
}

}  // namespace gdn
