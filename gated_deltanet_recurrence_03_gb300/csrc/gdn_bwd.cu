// Backward pass of the gated delta-rule recurrence: gradients of (out, S_final) with respect to q, k,
// v, g, beta and S0.  The forward is the token loop of "Transformer by Hand, ch. 7" (section "The
// formula", `delta_rule`), per sequence and value head with a_t = exp(g_t):
//     p = S^T k,   u = beta (v - a p),   S <- a S + k u^T,   o = scale S^T q.
// Walking it backwards with lam = dL/dS_t (from dL/dS_final):
//     lam += scale q do^T;   dq = scale (a S_{t-1} do + k (u.do));   du = lam^T k;   dk = lam u + S_{t-1} dp;
//     dv = beta du;   dbeta = du.(v - a p);   dp = -a beta du;   dg = a (<lam, S_{t-1}> - beta du.p);
//     lam <- a lam + k dp^T;   dS0 = lam at the sequence start.
// The value columns of S evolve independently, so one CTA owns one (sequence, value head, 32-column
// slice): warp w holds key rows R*w .. R*w+R-1 and lane j one column, state and adjoint in registers.
// The backward needs S_{t-1} in reverse order: a forward pass stores a checkpoint every kCk tokens;
// then, chunk by chunk from the end, the chunk's states are recomputed into a per-CTA scratch (about
// 64 MB over the whole grid, L2-resident) and walked backwards.  Sums over the value columns (dq, dk,
// dg, dbeta) are per-slice partials, added by a second kernel that also folds the GQA head groups.
// Token-serial on CUDA cores: a first path, not a tensor-core kernel.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kW = 32;         // value columns per CTA
constexpr int kCk = 16;        // tokens between checkpoints
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

template <int DK>
struct BwdSmem {
    float q[2][DK], k[2][DK];       // staged token (double buffered)
    float v[2][kW], dout[2][kW];
    float a[2], beta[2];
    float red_p[kWarps][kW], red_d[kWarps][kW];
    float wsum[kWarps];
    float csum[3];
};

// Stage token `tok` of value head h (query/key head hk) into buffer `buf`.  Needs q and dout only for
// backward steps.
template <typename T, int DK>
__device__ __forceinline__ void stage(BwdSmem<DK>& s, int buf, const T* q, const T* k, const T* v, const T* g,
                                      const T* beta, const T* dout, long long tok, int h, int hk, int Hqk, int Hv,
                                      int dv, int col0, bool with_q) {
    const int tid = threadIdx.x;
    if (tid < DK) {
        s.k[buf][tid] = to_f32(k[(tok * Hqk + hk) * DK + tid]);
        if (with_q) s.q[buf][tid] = to_f32(q[(tok * Hqk + hk) * DK + tid]);
    } else if (tid < DK + kW) {
        const int j = tid - DK;
        s.v[buf][j] = to_f32(v[(tok * Hv + h) * dv + col0 + j]);
        if (with_q) s.dout[buf][j] = to_f32(dout[(tok * Hv + h) * dv + col0 + j]);
    } else if (tid == DK + kW) {
        s.a[buf] = __expf(to_f32(g[tok * Hv + h]));
        s.beta[buf] = to_f32(beta[tok * Hv + h]);
    }
}

// One forward step on the thread's rows: p_j = sum_i S[i] k_i over the whole column, then the write.
template <int DK>
__device__ __forceinline__ void forward_step(float (&S)[DK / kWarps], BwdSmem<DK>& s, int buf, int w, int j) {
    constexpr int R = DK / kWarps;
    float pp = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) pp = fmaf(S[i], s.k[buf][R * w + i], pp);
    s.red_p[w][j] = pp;
    __syncthreads();
    float p = 0.f;
#pragma unroll
    for (int x = 0; x < kWarps; ++x) p += s.red_p[x][j];
    const float a = s.a[buf];
    const float u = s.beta[buf] * (s.v[buf][j] - a * p);
#pragma unroll
    for (int i = 0; i < R; ++i) S[i] = fmaf(a, S[i], s.k[buf][R * w + i] * u);
}

// Sum of v[i] over the 32 lanes for every row i < R, by halving: after the call lane `lane` holds the
// total of row row_of_lane<R>(lane) (all lanes hold one; several hold the same row).
template <int R>
__device__ __forceinline__ float row_reduce(float (&v)[R], int lane) {
    int m = 16;
#pragma unroll
    for (int n = R; n > 1; n >>= 1, m >>= 1) {
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = up ? v[i + n / 2] : v[i];
            const float send = up ? v[i] : v[i + n / 2];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    float r = v[0];
    for (; m >= 1; m >>= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
    return r;
}
template <int R>
__device__ __forceinline__ int row_of_lane(int lane) {
    int row = 0, m = 16;
#pragma unroll
    for (int n = R; n > 1; n >>= 1, m >>= 1)
        if (lane & m) row += n / 2;
    return row;
}
// The one lane per row that writes it: the lane bits below the halving masks are zero.
template <int R>
__device__ __forceinline__ bool row_writer(int lane) {
    int m = 16;
#pragma unroll
    for (int n = R; n > 1; n >>= 1) m >>= 1;
    return (lane & (2 * m - 1)) == 0;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

template <typename T, int DK>
__global__ void __launch_bounds__(kThreads)
bwd_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const T* __restrict__ g,
           const T* __restrict__ beta, const float* __restrict__ S0, const T* __restrict__ dout,
           const float* __restrict__ dS_final, float* __restrict__ part, float* __restrict__ grad_v,
           float* __restrict__ grad_S0, float* __restrict__ ckpt, float* __restrict__ scratch, int T_len, int Hqk,
           int Hv, int dv, const int32_t* __restrict__ cu, int nseq, float scale) {
    constexpr int R = DK / kWarps;
    __shared__ BwdSmem<DK> s;
    const int nsl = dv / kW;
    const int sl = blockIdx.x % nsl, h = (blockIdx.x / nsl) % Hv, seq = blockIdx.x / (nsl * Hv);
    if (seq >= nseq) return;
    const int hk = h / (Hv / Hqk), col0 = sl * kW;
    const int w = threadIdx.x >> 5, j = threadIdx.x & 31;
    long long t0, t1;
    seq_range(cu, seq, T_len, t0, t1);
    const long long len = t1 - t0;
    const long long nch = (len + kCk - 1) / kCk;
    // checkpoint slots of this sequence: slot(seq, c) = floor(t0 / kCk) + seq + c (no prefix sum needed)
    const long long slot0 = t0 / kCk + seq;
    const size_t slice = (size_t)DK * kW;
    const auto ck = [&](long long c) { return ckpt + (((slot0 + c) * Hv + h) * nsl + sl) * slice; };
    float* scr = scratch + (size_t)blockIdx.x * kCk * slice;
    const size_t state_base = ((size_t)seq * Hv + h) * DK * dv + col0 + j;   // element (row 0, column j)

    float S[R];
#pragma unroll
    for (int i = 0; i < R; ++i) S[i] = S0 ? S0[state_base + (size_t)(R * w + i) * dv] : 0.f;

    // ---- forward pass: checkpoint every kCk tokens
    int buf = 0;
    for (long long t = t0; t < t1; ++t, buf ^= 1) {
        if ((t - t0) % kCk == 0) {
            float* c = ck((t - t0) / kCk);
#pragma unroll
            for (int i = 0; i < R; ++i) c[(R * w + i) * kW + j] = S[i];
        }
        stage<T, DK>(s, buf, q, k, v, g, beta, dout, t, h, hk, Hqk, Hv, dv, col0, false);
        __syncthreads();
        forward_step<DK>(S, s, buf, w, j);
    }

    // ---- backward pass, chunk by chunk from the end
    float lam[R];
#pragma unroll
    for (int i = 0; i < R; ++i) lam[i] = dS_final ? dS_final[state_base + (size_t)(R * w + i) * dv] : 0.f;
    const int my_row = row_of_lane<R>(j);
    const bool writer = row_writer<R>(j);
    for (long long c = nch - 1; c >= 0; --c) {
        const long long tc0 = t0 + c * kCk, tc1 = min(t1, tc0 + kCk);
        const float* cs = ck(c);
#pragma unroll
        for (int i = 0; i < R; ++i) S[i] = cs[(R * w + i) * kW + j];
        for (long long t = tc0; t < tc1; ++t, buf ^= 1) {   // recompute the chunk's states S_{t-1}
            float* d = scr + (t - tc0) * slice;
#pragma unroll
            for (int i = 0; i < R; ++i) d[(R * w + i) * kW + j] = S[i];
            stage<T, DK>(s, buf, q, k, v, g, beta, dout, t, h, hk, Hqk, Hv, dv, col0, false);
            __syncthreads();
            forward_step<DK>(S, s, buf, w, j);
        }
        for (long long t = tc1 - 1; t >= tc0; --t, buf ^= 1) {
            const float* d = scr + (t - tc0) * slice;
            float Sp[R];
#pragma unroll
            for (int i = 0; i < R; ++i) Sp[i] = d[(R * w + i) * kW + j];
            stage<T, DK>(s, buf, q, k, v, g, beta, dout, t, h, hk, Hqk, Hv, dv, col0, true);
            __syncthreads();
            const float a = s.a[buf], bt = s.beta[buf], doj = s.dout[buf][j], vj = s.v[buf][j];
            const float* kk = s.k[buf];
            const float* qq = s.q[buf];
            float pp = 0.f, dd = 0.f;
#pragma unroll
            for (int i = 0; i < R; ++i) {
                lam[i] = fmaf(scale * qq[R * w + i], doj, lam[i]);
                pp = fmaf(Sp[i], kk[R * w + i], pp);
                dd = fmaf(lam[i], kk[R * w + i], dd);
            }
            s.red_p[w][j] = pp;
            s.red_d[w][j] = dd;
            __syncthreads();
            float p = 0.f, du = 0.f;
#pragma unroll
            for (int x = 0; x < kWarps; ++x) {
                p += s.red_p[x][j];
                du += s.red_d[x][j];
            }
            const float r = vj - a * p;
            const float u = bt * r;
            const float dp = -a * bt * du;
            float rq[R], rk[R], ls = 0.f;
#pragma unroll
            for (int i = 0; i < R; ++i) {
                rq[i] = a * Sp[i] * doj;
                rk[i] = fmaf(lam[i], u, Sp[i] * dp);
                ls = fmaf(lam[i], Sp[i], ls);
            }
            ls = warp_sum(ls);
            if (w == 0) {
                const float cb = warp_sum(du * r), ca = warp_sum(-bt * du * p), cu_ = warp_sum(u * doj);
                if (j == 0) {
                    s.csum[0] = cb;
                    s.csum[1] = ca;
                    s.csum[2] = cu_;
                }
            }
            if (j == 0) s.wsum[w] = ls;
            const float q_row = row_reduce<R>(rq, j);
            const float k_row = row_reduce<R>(rk, j);
            __syncthreads();
            float da = s.csum[1];
#pragma unroll
            for (int x = 0; x < kWarps; ++x) da += s.wsum[x];
            float* pr = part + (((size_t)t * Hv + h) * nsl + sl) * (2 * DK + 2);
            if (writer) {
                const int row = R * w + my_row;
                pr[row] = scale * fmaf(kk[row], s.csum[2], q_row);
                pr[DK + row] = k_row;
            }
            if (threadIdx.x == 0) {
                pr[2 * DK] = a * da;
                pr[2 * DK + 1] = s.csum[0];
            }
            if (w == 0) grad_v[((size_t)t * Hv + h) * dv + col0 + j] = bt * du;
#pragma unroll
            for (int i = 0; i < R; ++i) lam[i] = fmaf(a, lam[i], kk[R * w + i] * dp);
        }
    }
    if (grad_S0) {
#pragma unroll
        for (int i = 0; i < R; ++i) grad_S0[state_base + (size_t)(R * w + i) * dv] = lam[i];
    }
}

// Sum the per-slice partials: dq, dk of query/key head hk over its value heads and slices; dg, dbeta
// of value head h over its slices.  One block per token.
template <int DK>
__global__ void __launch_bounds__(256)
bwd_reduce_kernel(const float* __restrict__ part, float* __restrict__ grad_q, float* __restrict__ grad_k,
                  float* __restrict__ grad_g, float* __restrict__ grad_beta, int Hqk, int Hv, int nsl) {
    const long long tok = blockIdx.x;
    const int G = Hv / Hqk;
    const size_t stride = 2 * DK + 2;
    for (int idx = threadIdx.x; idx < Hqk * DK; idx += blockDim.x) {
        const int hk = idx / DK, i = idx % DK;
        float sq = 0.f, sk = 0.f;
        for (int h = hk * G; h < (hk + 1) * G; ++h)
            for (int sl = 0; sl < nsl; ++sl) {
                const float* pr = part + ((tok * Hv + h) * nsl + sl) * stride;
                sq += pr[i];
                sk += pr[DK + i];
            }
        grad_q[(tok * Hqk + hk) * DK + i] = sq;
        grad_k[(tok * Hqk + hk) * DK + i] = sk;
    }
    for (int h = threadIdx.x; h < Hv; h += blockDim.x) {
        float sg = 0.f, sb = 0.f;
        for (int sl = 0; sl < nsl; ++sl) {
            const float* pr = part + ((tok * Hv + h) * nsl + sl) * stride;
            sg += pr[2 * DK];
            sb += pr[2 * DK + 1];
        }
        grad_g[tok * Hv + h] = sg;
        grad_beta[tok * Hv + h] = sb;
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <typename T, int DK>
cudaError_t launch_typed(const BackwardArgs& a, const BwdLayout& L) {
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    float* ckpt = reinterpret_cast<float*>(ws + L.ckpt_off);
    float* scratch = reinterpret_cast<float*>(ws + L.scratch_off);
    float* part = reinterpret_cast<float*>(ws + L.part_off);
    const int nsl = a.dv / kW;
    bwd_kernel<T, DK><<<(unsigned)(a.num_seqs * a.Hv * nsl), kThreads, 0, a.stream>>>(
        static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
        static_cast<const T*>(a.g), static_cast<const T*>(a.beta), a.S0, static_cast<const T*>(a.dout),
        a.dS_final, part, a.grad_v, a.grad_S0, ckpt, scratch, a.T, a.Hqk, a.Hv, a.dv, a.cu_seqlens, a.num_seqs,
        a.scale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long ttot = a.cu_seqlens ? (long long)a.T : (long long)a.B * a.T;
    if (ttot > 0) {
        bwd_reduce_kernel<DK><<<(unsigned)ttot, 256, 0, a.stream>>>(part, a.grad_q, a.grad_k, a.grad_g, a.grad_beta,
                                                                     a.Hqk, a.Hv, nsl);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

BwdLayout backward_layout(int B, int T, int Hv, int dk, int dv, int nseq, bool packed) {
    const long long ttot = packed ? (long long)T : (long long)B * T;
    const int nsl = dv / kW;
    const size_t slice = (size_t)dk * kW * sizeof(float);
    const long long slots = (ttot + kCk - 1) / kCk + nseq;
    BwdLayout L{};
    L.ckpt_off = 0;
    L.scratch_off = align256(L.ckpt_off + (size_t)slots * Hv * nsl * slice);
    L.part_off = align256(L.scratch_off + (size_t)nseq * Hv * nsl * kCk * slice);
    L.total = align256(L.part_off + (size_t)ttot * Hv * nsl * (2 * dk + 2) * sizeof(float));
    return L;
}

cudaError_t launch_backward(const BackwardArgs& a) {
    const BwdLayout L = backward_layout(a.B, a.T, a.Hv, a.dk, a.dv, a.num_seqs, a.cu_seqlens != nullptr);
    const bool bf = a.dtype == GDN_BF16;
    switch (a.dk) {
        case 32: return bf ? launch_typed<__nv_bfloat16, 32>(a, L) : launch_typed<float, 32>(a, L);
        case 64: return bf ? launch_typed<__nv_bfloat16, 64>(a, L) : launch_typed<float, 64>(a, L);
        case 128: return bf ? launch_typed<__nv_bfloat16, 128>(a, L) : launch_typed<float, 128>(a, L);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
