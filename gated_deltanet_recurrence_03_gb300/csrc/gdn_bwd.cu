// Backward pass of the gated delta-rule recurrence: gradients of (out, S_final) with respect to q, k,
// v, g, beta and S0.  The forward is the token loop of "Transformer by Hand, ch. 7" (section "The
// formula", `delta_rule`), per sequence and value head with a_t = exp(g_t):
//     p = S^T k,   u = beta (v - a p),   S <- a S + k u^T,   o = scale S^T q.
// The gradient is taken through the chunked form of that loop (chunk length C = 64, zero-padded at a
// sequence end, which leaves the state unchanged).  Inside a chunk, with G_r = sum_{s<=r} g_s,
// D_rs = exp(G_r - G_s) for s <= r, gamma = exp(G), S the state at the chunk start:
//     A = strict lower part of D o (K K^T),    T = (I + diag(beta) A)^{-1},
//     W = T diag(beta gamma) K,   U~ = T diag(beta) V,   U = U~ - W S,
//     P = scale D o (Q K^T) (s <= r),   O = scale diag(gamma) Q S + P U,
//     S' = gamma_C S + K~^T U,   K~ = diag(gamma_C / gamma) K.
// Its adjoint, for dO and lam = dL/dS' given:
//     dU = K~ lam + P^T dO,   dL/dS = gamma_C lam + scale Q^T diag(gamma) dO - W^T dU,
// and the chunk-local gradients follow by the chain rule through T (dT -> -T^T dT T^T), the decay
// ratios (d exp(G_r - G_s) adds to G_r and subtracts from G_s) and dg = reverse cumulative sum of dG.
//
// Four kernels, all in fp32 accuracy, their products on tf32 tensor cores with each fp32 operand split
// into two tf32 parts (the WY kernel's triangular solve on CUDA cores; for bf16 inputs with
// dk = dv = 128 the two chains run instead as the tcgen05 kernels of gdn_bwd_tc.cu):
//   bwd_wy_kernel         per (chunk, query/key head): T, W, U~, P and G of each of its value heads
//   bwd_state_fwd_kernel  per (sequence, value head, column slice): chunk-start states S, and U
//   bwd_state_adj_kernel  per (sequence, value head, column slice), chunks in reverse: lam, dU, dS0
//   bwd_local_kernel      per (chunk, query/key head): dq, dk (summed over its value heads), dv, dg, dbeta
// Chunks of sequence i occupy workspace slots floor(t0_i / C) + i + c, so no prefix sum is needed.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kC = 64;      // chunk length
constexpr int kLCC = kC + 4; // C x C matrices in shared memory: rows 4 banks apart (conflict-free fragments)

// ---------------------------------------------------------------- register tiles
template <int RM, int CN>
__device__ __forceinline__ void tile_zero(float (&acc)[RM][CN]) {
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int m = 0; m < CN; ++m) acc[i][m] = 0.f;
}

// ---------------------------------------------------------------- tensor-core products in fp32 accuracy
// mma.sync m16n8k8 with tf32 operands; each fp32 operand is split as x = hi + lo and
// a b ~ hi_a hi_b + hi_a lo_b + lo_a hi_b (the error-corrected tf32 product of Ootomo and Yokota,
// 2022).  hi is x rounded to tf32's 10 fraction bits, to nearest with ties away from zero, on the
// bit pattern: half a tf32 ulp (bit 12) is added and the 13 low bits cleared, integer operations
// only (a conversion instruction per element throttled the kernels).  lo = x - hi is exact in fp32
// and at most half a tf32 ulp of x; it is passed as it is, and the tensor core reads its 19 high bits
// (a truncation of at most 2^-10 of lo), so the error of hi + lo is below 2^-21 |x| and the dropped
// lo_a lo_b term about 2^-22 of the product.  Fragment coordinates (g = lane / 4, t = lane % 4):
// A (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4); B (k = t, n = g), (k = t + 4, n = g); accumulator
// (g, 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1).
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    hi = (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
    lo = __float_as_uint(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma_3xtf32(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                           const uint32_t (&bh)[2], const uint32_t (&bl)[2]) {
    mma_tf32(d, al, bh);
    mma_tf32(d, ah, bl);
    mma_tf32(d, ah, bh);
}
// Operands whose values tf32 represents exactly (bf16 inputs widened to fp32: K, Q, dO, V) have a zero
// lo part, so their lo products are skipped: EA / EB mark A / B exact (three, two or one MMA).
template <bool EA, bool EB>
__device__ __forceinline__ void mma_split(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                          const uint32_t (&bh)[2], const uint32_t (&bl)[2]) {
    if (!EA) mma_tf32(d, al, bh);
    if (!EB) mma_tf32(d, ah, bl);
    mma_tf32(d, ah, bh);
}
// Split x into tf32 hi / lo, or, for an exact operand, take its bits as they are (lo unused).
template <bool EXACT>
__device__ __forceinline__ void split_x(float x, uint32_t& hi, uint32_t& lo) {
    if (EXACT) hi = __float_as_uint(x);
    else split_tf32(x, hi, lo);
}
// A fragment: rows row0 + g (+ 8), columns k0 + t (+ 4) of a row-major fp32 matrix.
template <bool EXACT = false>
__device__ __forceinline__ void frag_a(const float* A, int ld, int row0, int k0, int g, int t, uint32_t (&hi)[4],
                                       uint32_t (&lo)[4]) {
    split_x<EXACT>(A[(row0 + g) * ld + k0 + t], hi[0], lo[0]);
    split_x<EXACT>(A[(row0 + g + 8) * ld + k0 + t], hi[1], lo[1]);
    split_x<EXACT>(A[(row0 + g) * ld + k0 + t + 4], hi[2], lo[2]);
    split_x<EXACT>(A[(row0 + g + 8) * ld + k0 + t + 4], hi[3], lo[3]);
}
// B fragment of B = X^T (B[k][n] = X[n][k], X row-major): n = n0 + g, k = k0 + t (+ 4).
template <bool EXACT = false>
__device__ __forceinline__ void frag_bt(const float* X, int ld, int n0, int k0, int g, int t, uint32_t (&hi)[2],
                                        uint32_t (&lo)[2]) {
    split_x<EXACT>(X[(n0 + g) * ld + k0 + t], hi[0], lo[0]);
    split_x<EXACT>(X[(n0 + g) * ld + k0 + t + 4], hi[1], lo[1]);
}
// A fragment of A stored k-major (A[m][k] = X[k][m]): rows row0 + g (+ 8), k = k0 + t (+ 4).
template <bool EXACT = false>
__device__ __forceinline__ void frag_at(const float* X, int ld, int row0, int k0, int g, int t, uint32_t (&hi)[4],
                                        uint32_t (&lo)[4]) {
    split_x<EXACT>(X[(k0 + t) * ld + row0 + g], hi[0], lo[0]);
    split_x<EXACT>(X[(k0 + t) * ld + row0 + g + 8], hi[1], lo[1]);
    split_x<EXACT>(X[(k0 + t + 4) * ld + row0 + g], hi[2], lo[2]);
    split_x<EXACT>(X[(k0 + t + 4) * ld + row0 + g + 8], hi[3], lo[3]);
}
// A fragment of a row-major A with column k scaled by ks[k] (A diag(ks)).
__device__ __forceinline__ void frag_a_scaled(const float* A, int ld, const float* ks, int row0, int k0, int g, int t,
                                              uint32_t (&hi)[4], uint32_t (&lo)[4]) {
    const float s0 = ks[k0 + t], s1 = ks[k0 + t + 4];
    split_tf32(s0 * A[(row0 + g) * ld + k0 + t], hi[0], lo[0]);
    split_tf32(s0 * A[(row0 + g + 8) * ld + k0 + t], hi[1], lo[1]);
    split_tf32(s1 * A[(row0 + g) * ld + k0 + t + 4], hi[2], lo[2]);
    split_tf32(s1 * A[(row0 + g + 8) * ld + k0 + t + 4], hi[3], lo[3]);
}
// The same with column k of A (row k of X) scaled by ks[k] (a diagonal matrix between the factors).
__device__ __forceinline__ void frag_at_scaled(const float* X, int ld, const float* ks, int row0, int k0, int g, int t,
                                               uint32_t (&hi)[4], uint32_t (&lo)[4]) {
    const float s0 = ks[k0 + t], s1 = ks[k0 + t + 4];
    split_tf32(s0 * X[(k0 + t) * ld + row0 + g], hi[0], lo[0]);
    split_tf32(s0 * X[(k0 + t) * ld + row0 + g + 8], hi[1], lo[1]);
    split_tf32(s1 * X[(k0 + t + 4) * ld + row0 + g], hi[2], lo[2]);
    split_tf32(s1 * X[(k0 + t + 4) * ld + row0 + g + 8], hi[3], lo[3]);
}
// B fragment of B stored k-major (B[k][n] = X[k][n]): n = n0 + g, k = k0 + t (+ 4).
template <bool EXACT = false>
__device__ __forceinline__ void frag_b(const float* X, int ld, int n0, int k0, int g, int t, uint32_t (&hi)[2],
                                       uint32_t (&lo)[2]) {
    split_x<EXACT>(X[(k0 + t) * ld + n0 + g], hi[0], lo[0]);
    split_x<EXACT>(X[(k0 + t + 4) * ld + n0 + g], hi[1], lo[1]);
}
// acc[q] += A B over k < K for the 16 rows from row0 and the NT n-tiles of 8 from nb0, in fp32 accuracy
// (three-product tf32 split).  AT: A stored k-major; BT: B stored n-major (X[n][k]).
template <int NT, int K, bool AT, bool BT, bool EA = false, bool EB = false>
__device__ __forceinline__ void mma_prod(float (&acc)[NT][4], const float* A, int lda, const float* B, int ldb,
                                         int row0, int nb0, int g, int t) {
#pragma unroll 2
    for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t ah[4], al[4];
        if (AT) frag_at<EA>(A, lda, row0, k0, g, t, ah, al);
        else frag_a<EA>(A, lda, row0, k0, g, t, ah, al);
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            uint32_t bh[2], bl[2];
            if (BT) frag_bt<EB>(B, ldb, 8 * (nb0 + q), k0, g, t, bh, bl);
            else frag_b<EB>(B, ldb, 8 * (nb0 + q), k0, g, t, bh, bl);
            mma_split<EA, EB>(acc[q], ah, al, bh, bl);
        }
    }
}
// The same with column k of A scaled by as[k] (A diag(as) B: a diagonal between the factors), A fp32.
template <int NT, int K, bool AT, bool EB = false>
__device__ __forceinline__ void mma_prod_as(float (&acc)[NT][4], const float* A, int lda, const float* as,
                                            const float* B, int ldb, int row0, int nb0, int g, int t) {
#pragma unroll 2
    for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t ah[4], al[4];
        if (AT) frag_at_scaled(A, lda, as, row0, k0, g, t, ah, al);
        else frag_a_scaled(A, lda, as, row0, k0, g, t, ah, al);
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            uint32_t bh[2], bl[2];
            frag_b<EB>(B, ldb, 8 * (nb0 + q), k0, g, t, bh, bl);
            mma_split<false, EB>(acc[q], ah, al, bh, bl);
        }
    }
}
// sign * (N accumulator fragments of rows row0 .. row0 + 15, n-tiles nb0 .. nb0 + N - 1) to D.
template <int N>
__device__ __forceinline__ void store_frag(float* D, int ld, const float (&f)[N][4], int row0, int nb0, int g, int t,
                                           float sign) {
#pragma unroll
    for (int q = 0; q < N; ++q) {
        const int c = 8 * (nb0 + q) + 2 * t;
        D[(row0 + g) * ld + c] = sign * f[q][0];
        D[(row0 + g) * ld + c + 1] = sign * f[q][1];
        D[(row0 + g + 8) * ld + c] = sign * f[q][2];
        D[(row0 + g + 8) * ld + c + 1] = sign * f[q][3];
    }
}

// 16 bytes of fp32 or bf16 values as fp32 (bf16 -> fp32 is a 16-bit shift).
__device__ __forceinline__ void unpack16(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack16(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Rows [0, ROWS) x columns [0, WIDTH) of an element-type block (global row stride `stride` elements;
// rows >= n read as zero) into shared memory as fp32 with leading dimension `ld`.  With `vec` (the
// source 16-byte aligned; strides and widths are multiples of 16 bytes) every thread issues all of
// its 16-byte loads before its stores.
template <typename TT, int ROWS, int WIDTH, int NT>
__device__ __forceinline__ void ld_in(float* __restrict__ dst, int ld, const TT* __restrict__ src, size_t stride,
                                      int n, int tid, bool vec) {
    constexpr int EPV = 16 / (int)sizeof(TT), V = WIDTH / EPV, TOTAL = ROWS * V, PER = (TOTAL + NT - 1) / NT;
    if (vec) {
        uint4 b[PER];
#pragma unroll
        for (int p = 0; p < PER; ++p) {
            const int idx = tid + p * NT, r = idx / V;
            b[p] = make_uint4(0u, 0u, 0u, 0u);
            if ((TOTAL % NT == 0 || idx < TOTAL) && r < n)
                b[p] = *reinterpret_cast<const uint4*>(src + (size_t)r * stride + (idx % V) * EPV);
        }
#pragma unroll
        for (int p = 0; p < PER; ++p) {
            const int idx = tid + p * NT;
            if (TOTAL % NT == 0 || idx < TOTAL) {
                float f[EPV];
                unpack16(b[p], f);
                float* d = dst + (idx / V) * ld + (idx % V) * EPV;
#pragma unroll
                for (int x = 0; x < EPV; ++x) d[x] = f[x];
            }
        }
    } else {
        for (int idx = tid; idx < ROWS * WIDTH; idx += NT) {
            const int r = idx / WIDTH, j = idx % WIDTH;
            dst[r * ld + j] = r < n ? to_f32(src[(size_t)r * stride + j]) : 0.f;
        }
    }
}

// Same for fp32 workspace blocks (always 16-byte aligned, all rows valid).
template <int ROWS, int WIDTH, int NT>
__device__ __forceinline__ void ld_ws(float* __restrict__ dst, int ld, const float* __restrict__ src, size_t stride,
                                      int tid) {
    ld_in<float, ROWS, WIDTH, NT>(dst, ld, src, stride, ROWS, tid, true);
}

// Workspace slot of chunk 0 of sequence i.
__device__ __forceinline__ long long slot_base(const int32_t* cu, int i, int T) {
    long long t0, t1;
    seq_range(cu, i, T, t0, t1);
    return t0 / kC + i;
}

// The (sequence, first token, valid rows) of a workspace slot, or false for a slot that holds no chunk.
__device__ __forceinline__ bool slot_chunk(const int32_t* cu, int nseq, int T, long long slot, int& seq,
                                           long long& tok0, int& n) {
    int lo = 0, hi = nseq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (slot_base(cu, mid, T) <= slot) lo = mid;
        else hi = mid - 1;
    }
    long long t0, t1;
    seq_range(cu, lo, T, t0, t1);
    const long long c = slot - (t0 / kC + lo);
    if (c < 0 || t0 + c * kC >= t1) return false;
    seq = lo;
    tok0 = t0 + c * kC;
    n = (int)min((long long)kC, t1 - tok0);
    return true;
}

// Per-(slot, value head) workspace arrays.
struct Ws {
    float *T, *P, *W, *U, *G, *S, *dS, *dU, *R;   // R: per-row l2 scalars of K and Q (prefill front end)
};

template <int DK, int DV>
struct WsDims {
    static constexpr size_t T = (size_t)kC * kC, P = (size_t)kC * kC, W = (size_t)kC * DK, U = (size_t)kC * DV,
                            G = kC, S = (size_t)DK * DV, dS = (size_t)DK * DV, dU = (size_t)kC * DV, R = 2 * kC;
};

// Fragment coordinates of accumulator element e of n-tile nb: row row0 + g (+ 8 for e >= 2),
// column 8 nb + 2 t + (e & 1).
__device__ __forceinline__ int frow(int row0, int g, int e) { return row0 + g + (e >= 2 ? 8 : 0); }
__device__ __forceinline__ int fcol(int nb, int t, int e) { return 8 * nb + 2 * t + (e & 1); }

// An M x N product over the 8 warps: the M / 16 row tiles first, the N / 8 column tiles split among
// the warps that share a row tile.  Warp w: row tile w % MT, column tiles (w / MT) NT .. + NT - 1.
template <int M, int N>
struct ChainTiles {
    static constexpr int MT = M / 16, WPM = 8 / MT, NT = (N / 8) / WPM;
    static_assert(MT >= 1 && MT <= 8 && 8 % MT == 0 && (N / 8) % WPM == 0 && NT >= 1, "tile split");
};

// ---------------------------------------------------------------- kernel 1: WY factors per chunk
constexpr int kWyThreads = 256;

// Shared memory of the WY kernel: about 106 KB at dk = dv = 128, so that two CTAs fit on an SM.  Q and
// V are staged half their columns at a time; Q K^T lives in the L buffer (P of every value head is
// formed before the first L).
template <int DK, int DV>
struct WySmem {
    static constexpr int DH = (DK > DV ? DK : DV) / 2;   // staged columns of Q or V
    static constexpr int LK = DK + 4, LQV = DH + 4;
    static constexpr int K_ = 0, QV_ = K_ + kC * LK, KK_ = QV_ + kC * LQV, L_ = KK_ + kC * kLCC,
                         T_ = L_ + kC * kLCC, Y_ = T_ + kC * kLCC, VEC_ = Y_ + 3 * 256;
    static constexpr int FLOATS = VEC_ + 6 * kC;
    static constexpr size_t BYTES = (size_t)FLOATS * 4;
};

// sum over the WIDTH columns of x_i^2 added to r[i] (one warp per row).
template <int ROWS, int WIDTH, int NWARPS>
__device__ __forceinline__ void row_sumsq_add(const float* __restrict__ x, int ld, float* __restrict__ r, int warp,
                                              int lane) {
    for (int i = warp; i < ROWS; i += NWARPS) {
        float s = 0.f;
        for (int c = lane; c < WIDTH; c += 32) s = fmaf(x[i * ld + c], x[i * ld + c], s);
#pragma unroll
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) r[i] += s;
    }
}

// With A_log non-null, g and beta hold the raw projections a, b and the gates are formed on load;
// with normalize, q and k are l2-normalised through per-row scalars (the prefill's front end).
template <typename TT, int DK, int DV>
__global__ void __launch_bounds__(kWyThreads, 2)
bwd_wy_kernel(const TT* __restrict__ q, const TT* __restrict__ k, const TT* __restrict__ v, const TT* __restrict__ g,
              const TT* __restrict__ beta, Ws ws, int T_len, int Hqk, int Hv, const int32_t* __restrict__ cu,
              int nseq, float scale, bool vec, const float* __restrict__ A_log, const float* __restrict__ dt_bias,
              bool normalize) {
    using L = WySmem<DK, DV>;
    using D = WsDims<DK, DV>;
    constexpr int QH = DK / 2, VH = DV / 2;   // columns of Q and of V per staged half
    extern __shared__ __align__(16) float sm[];
    float* sK = sm + L::K_;
    float* sQV = sm + L::QV_;
    float* sKK = sm + L::KK_;
    float* sQK = sm + L::L_;   // Q K^T until P of every value head is out, then L
    float* sL = sm + L::L_;
    float* sT = sm + L::T_;
    float* sY = sm + L::Y_;   // off-diagonal block sums of the solve: up to 3 blocks of 16 x 16
    float* sG = sm + L::VEC_;
    float* sBeta = sG + kC;
    float* sBG = sBeta + kC;
    float* sGraw = sBG + kC;
    float* sRK = sGraw + kC;   // per-row l2 scalars of K and Q (1 without normalisation)
    float* sRQ = sRK + kC;

    const long long slot = blockIdx.x;
    const int hk = blockIdx.y, G = Hv / Hqk;
    int seq, n;
    long long tok0;
    if (!slot_chunk(cu, nseq, T_len, slot, seq, tok0, n)) return;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, lg = lane / 4, lt = lane % 4;   // fragment (g, t)
    constexpr bool kEx = sizeof(TT) == 2;   // bf16 K, Q, V are exact in tf32
    const TT* qrow = q + (tok0 * Hqk + hk) * DK;

    ld_in<TT, kC, DK, kWyThreads>(sK, L::LK, k + (tok0 * Hqk + hk) * DK, (size_t)Hqk * DK, n, tid, vec);
    ld_in<TT, kC, QH, kWyThreads>(sQV, L::LQV, qrow, (size_t)Hqk * DK, n, tid, vec);
    if (tid < kC) {
        sRK[tid] = normalize ? 0.f : 1.f;
        sRQ[tid] = normalize ? 0.f : 1.f;
    }
    __syncthreads();
    // Gram matrices K K^T and Q K^T on tensor cores (both operands exact in tf32 for bf16 inputs); Q K^T
    // over the two column halves of Q in turn
    using TG = ChainTiles<kC, kC>;
    float kk[TG::NT][4], qk[TG::NT][4];
    tile_zero(kk);
    tile_zero(qk);
    const int gm = 16 * (warp % TG::MT), gn = (warp / TG::MT) * TG::NT;
    if (normalize) {
        row_sumsq_add<kC, DK, kWyThreads / 32>(sK, L::LK, sRK, warp, lane);
        row_sumsq_add<kC, QH, kWyThreads / 32>(sQV, L::LQV, sRQ, warp, lane);
    }
    mma_prod<TG::NT, DK, false, true, kEx, kEx>(kk, sK, L::LK, sK, L::LK, gm, gn, lg, lt);
    mma_prod<TG::NT, QH, false, true, kEx, kEx>(qk, sQV, L::LQV, sK, L::LK, gm, gn, lg, lt);
    __syncthreads();
    ld_in<TT, kC, QH, kWyThreads>(sQV, L::LQV, qrow + QH, (size_t)Hqk * DK, n, tid, vec);
    __syncthreads();
    if (normalize) row_sumsq_add<kC, QH, kWyThreads / 32>(sQV, L::LQV, sRQ, warp, lane);
    mma_prod<TG::NT, QH, false, true, kEx, kEx>(qk, sQV, L::LQV, sK + QH, L::LK, gm, gn, lg, lt);
    store_frag<TG::NT>(sKK, kLCC, kk, gm, gn, lg, lt, 1.f);
    store_frag<TG::NT>(sQK, kLCC, qk, gm, gn, lg, lt, 1.f);
    __syncthreads();
    if (normalize && tid < kC) {
        sRK[tid] = rsqrtf(sRK[tid] + 1e-6f);
        sRQ[tid] = rsqrtf(sRQ[tid] + 1e-6f);
    }

    // The gates of value head h and G = their inclusive prefix sum (lane l of warp 0: tokens 2l, 2l + 1).
    const auto head_gates = [&](int h) {
        if (tid < kC) {
            const bool ok = tid < n;
            float gt = ok ? to_f32(g[(tok0 + tid) * Hv + h]) : 0.f;
            float bt = ok ? to_f32(beta[(tok0 + tid) * Hv + h]) : 0.f;
            if (A_log && ok) gates_from_raw(gt, bt, A_log[h], dt_bias[h], gt, bt);   // rows past n stay 0
            sGraw[tid] = gt;
            sBeta[tid] = bt;
        }
        __syncthreads();
        if (tid < 32) {
            const float a = sGraw[2 * tid], b = sGraw[2 * tid + 1];
            float x = a + b;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (tid >= o) x += y;
            }
            sG[2 * tid] = x - b;
            sG[2 * tid + 1] = x;
        }
        __syncthreads();
    };

    // P = scale D o QK^T (s <= r) of every value head to the workspace, with G and the l2 scalars
    for (int j = 0; j < G; ++j) {
        const int h = hk * G + j;
        const size_t wi = (size_t)slot * Hv + h;
        head_gates(h);
        if (tid < kC) {
            ws.G[wi * D::G + tid] = sG[tid];
            if (normalize) {   // for the chains, the output kernel and the chunk-local kernel
                ws.R[wi * D::R + tid] = sRK[tid];
                ws.R[wi * D::R + kC + tid] = sRQ[tid];
            }
        }
        for (int idx = tid; idx < kC * kC; idx += kWyThreads) {
            const int r = idx / kC, s = idx % kC;
            const float d = s <= r ? __expf(sG[r] - sG[s]) : 0.f;
            ws.P[wi * D::P + idx] = scale * d * (sRQ[r] * sRK[s]) * sQK[r * kLCC + s];
        }
        __syncthreads();   // sG of the next head; after the last, the Q K^T buffer is free for L
    }

    for (int j = 0; j < G; ++j) {
        const int h = hk * G + j;
        const size_t wi = (size_t)slot * Hv + h;
        head_gates(h);
        if (tid < kC) sBG[tid] = sBeta[tid] * __expf(sG[tid]) * sRK[tid];   // W = T diag(beta gamma) (diag(rk) K)
        // L = diag(beta) (D o KK^T) strictly below the diagonal
        for (int idx = tid; idx < kC * kC; idx += kWyThreads) {
            const int r = idx / kC, s = idx % kC;
            sL[r * kLCC + s] = s < r ? sBeta[r] * __expf(sG[r] - sG[s]) * (sRK[r] * sRK[s]) * sKK[r * kLCC + s] : 0.f;
        }
        __syncthreads();
        {   // T = (I + L)^{-1} in 16 x 16 blocks: each diagonal block by forward substitution (one thread
            // per column), then block row i below the diagonal from (I + L) T = I:
            //     T_ij = -T_ii sum_{l=j}^{i-1} L_il T_lj,   for i - j = 1, 2, 3 in turn.
            if (tid < kC) {
                const int o = 16 * (tid / 16), c = tid % 16;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float acc = r == c ? 1.f : 0.f;
#pragma unroll
                    for (int qq = 0; qq < r; ++qq) acc = fmaf(-sL[(o + r) * kLCC + o + qq], x[qq], acc);
                    x[r] = acc;
                    sT[(o + r) * kLCC + o + c] = acc;
                }
            } else {   // blocks above the diagonal are zero
                for (int idx = tid - kC; idx < 6 * 256; idx += kWyThreads - kC) {
                    const int blk = idx / 256, e = idx % 256;
                    const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2), bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                    sT[(16 * bi + e / 16) * kLCC + 16 * bj + e % 16] = 0.f;
                }
            }
            __syncthreads();
            for (int d = 1; d < 4; ++d) {
                const int nb = 4 - d;
                for (int idx = tid; idx < nb * 256; idx += kWyThreads) {
                    const int bj = idx / 256, e = idx % 256, r = e / 16, c = e % 16, bi = bj + d;
                    float acc = 0.f;
                    for (int bl = bj; bl < bi; ++bl)
#pragma unroll
                        for (int qq = 0; qq < 16; ++qq)
                            acc = fmaf(sL[(16 * bi + r) * kLCC + 16 * bl + qq], sT[(16 * bl + qq) * kLCC + 16 * bj + c], acc);
                    sY[idx] = acc;
                }
                __syncthreads();
                for (int idx = tid; idx < nb * 256; idx += kWyThreads) {
                    const int bj = idx / 256, e = idx % 256, r = e / 16, c = e % 16, bi = bj + d;
                    float acc = 0.f;
#pragma unroll
                    for (int qq = 0; qq < 16; ++qq)
                        acc = fmaf(sT[(16 * bi + r) * kLCC + 16 * bi + qq], sY[bj * 256 + qq * 16 + c], acc);
                    sT[(16 * bi + r) * kLCC + 16 * bj + c] = -acc;
                }
                __syncthreads();
            }
        }
        for (int idx = tid; idx < kC * kC; idx += kWyThreads) ws.T[wi * D::T + idx] = sT[(idx / kC) * kLCC + idx % kC];
        {   // W = T diag(beta gamma) K on tensor cores (K exact for bf16 inputs)
            using TW = ChainTiles<kC, DK>;
            float acc[TW::NT][4];
            tile_zero(acc);
            const int wm = 16 * (warp % TW::MT), wn = (warp / TW::MT) * TW::NT;
#pragma unroll 2
            for (int k0 = 0; k0 < kC; k0 += 8) {
                uint32_t ah[4], al[4];
                frag_a_scaled(sT, kLCC, sBG, wm, k0, lg, lt, ah, al);
#pragma unroll
                for (int qq = 0; qq < TW::NT; ++qq) {
                    uint32_t bh[2], bl[2];
                    frag_b<kEx>(sK, L::LK, 8 * (wn + qq), k0, lg, lt, bh, bl);
                    mma_split<false, kEx>(acc[qq], ah, al, bh, bl);
                }
            }
#pragma unroll
            for (int qq = 0; qq < TW::NT; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    ws.W[wi * D::W + (size_t)frow(wm, lg, e) * DK + fcol(wn + qq, lt, e)] = acc[qq][e];
        }
        // U~ = T diag(beta) V on tensor cores (V exact for bf16 inputs), over the two column halves of V
        for (int half = 0; half < 2; ++half) {
            ld_in<TT, kC, VH, kWyThreads>(sQV, L::LQV, v + (tok0 * Hv + h) * DV + half * VH, (size_t)Hv * DV, n, tid, vec);
            __syncthreads();
            using TV = ChainTiles<kC, VH>;
            float acc[TV::NT][4];
            tile_zero(acc);
            const int vm = 16 * (warp % TV::MT), vn = (warp / TV::MT) * TV::NT;
#pragma unroll 2
            for (int k0 = 0; k0 < kC; k0 += 8) {
                uint32_t ah[4], al[4];
                frag_a_scaled(sT, kLCC, sBeta, vm, k0, lg, lt, ah, al);
#pragma unroll
                for (int qq = 0; qq < TV::NT; ++qq) {
                    uint32_t bh[2], bl[2];
                    frag_b<kEx>(sQV, L::LQV, 8 * (vn + qq), k0, lg, lt, bh, bl);
                    mma_split<false, kEx>(acc[qq], ah, al, bh, bl);
                }
            }
#pragma unroll
            for (int qq = 0; qq < TV::NT; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    ws.U[wi * D::U + (size_t)frow(vm, lg, e) * DV + half * VH + fcol(vn + qq, lt, e)] = acc[qq][e];
            __syncthreads();   // sQV is refilled next (the other half of V, or the next head's V)
        }
    }
}

// ---------------------------------------------------------------- kernels 2 and 3: the chunk chains
// Both chains run their products on tf32 tensor cores with the three-product split (fp32 accuracy),
// 8 warps per CTA; each product's 16 x 8 output tiles are spread over the warps by ChainTiles.
constexpr int kStThreads = 256;

template <int DV>
constexpr int slice_width() { return DV < 64 ? DV : 64; }

template <int DK, int DV>
struct StSmem {
    // leading dimensions: width + 4 (= 4 mod 32: conflict-free row-major fragments)
    static constexpr int SW = slice_width<DV>(), LK = DK + 4, LCC = kC + 4, LS = SW + 4;
    // forward: W [C][DK], K [C][DK], U slice [C][SW], S slice [DK][SW]
    // adjoint: W, K, Q [C][DK], P [C][C], dO and dU slices [C][SW], lam slice [DK][SW]
    static constexpr int W_ = 0, K_ = W_ + kC * LK, Q_ = K_ + kC * LK, P_ = Q_ + kC * LK, X_ = P_ + kC * LCC,
                         Y_ = X_ + kC * LS, S_ = Y_ + kC * LS, G_ = S_ + DK * LS, R_ = G_ + kC;
    static constexpr int FLOATS = R_ + kC;
    static constexpr size_t BYTES = (size_t)FLOATS * 4;
    static_assert(K_ % 4 == 0 && Q_ % 4 == 0 && P_ % 4 == 0 && X_ % 4 == 0 && Y_ % 4 == 0 && S_ % 4 == 0,
                  "16-byte aligned regions");
};

// Chunk-start states S (to the workspace) and U = U~ - W S (over U~ in the workspace).  With normalize,
// the update reads K through its per-row l2 scalars (written by the WY kernel).
template <typename TT, int DK, int DV>
__global__ void __launch_bounds__(kStThreads)
bwd_state_fwd_kernel(const TT* __restrict__ k, const float* __restrict__ S0, float* __restrict__ S_final, Ws ws,
                     int T_len, int Hqk, int Hv, const int32_t* __restrict__ cu, int nseq, bool vec, bool normalize) {
    using L = StSmem<DK, DV>;
    using D = WsDims<DK, DV>;
    constexpr int SW = L::SW, NSL = DV / SW;
    using TU = ChainTiles<kC, SW>;   // U: C x SW
    using TS = ChainTiles<DK, SW>;   // S: DK x SW
    constexpr bool kEx = sizeof(TT) == 2;   // bf16 K is exact in tf32
    extern __shared__ __align__(16) float sm[];
    float* sW = sm + L::W_;
    float* sK = sm + L::K_;
    float* sU = sm + L::X_;
    float* sS = sm + L::S_;
    float* sG = sm + L::G_;
    float* sRK = sm + L::R_;   // per-row l2 scalars of K
    const int sl = blockIdx.x % NSL, h = (blockIdx.x / NSL) % Hv, seq = blockIdx.x / (NSL * Hv);
    if (seq >= nseq) return;
    const int hk = h / (Hv / Hqk), col0 = sl * SW;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, g = lane / 4, t = lane % 4;
    const int um = 16 * (warp % TU::MT), un = (warp / TU::MT) * TU::NT;
    const int sm0 = 16 * (warp % TS::MT), sn = (warp / TS::MT) * TS::NT;
    long long t0, t1;
    seq_range(cu, seq, T_len, t0, t1);
    const long long nch = (t1 - t0 + kC - 1) / kC, slot0 = t0 / kC + seq;
    const size_t sbase = ((size_t)seq * Hv + h) * DK * DV + col0;
    for (int idx = tid; idx < DK * SW; idx += kStThreads) {
        const int i = idx / SW, j = idx % SW;
        sS[i * L::LS + j] = S0 ? S0[sbase + (size_t)i * DV + j] : 0.f;
    }

    for (long long c = 0; c < nch; ++c) {
        const size_t wi = (size_t)(slot0 + c) * Hv + h;
        const long long tok0 = t0 + c * kC;
        const int n = (int)min((long long)kC, t1 - tok0);
        if (tid < kC) {
            sG[tid] = ws.G[wi * D::G + tid];
            sRK[tid] = normalize ? ws.R[wi * D::R + tid] : 1.f;
        }
        ld_ws<kC, DK, kStThreads>(sW, L::LK, ws.W + wi * D::W, DK, tid);
        ld_ws<kC, SW, kStThreads>(sU, L::LS, ws.U + wi * D::U + col0, DV, tid);
        ld_in<TT, kC, DK, kStThreads>(sK, L::LK, k + (tok0 * Hqk + hk) * DK, (size_t)Hqk * DK, n, tid, vec);
        __syncthreads();
        for (int idx = tid; idx < DK * SW; idx += kStThreads) {
            const int i = idx / SW, j = idx % SW;
            ws.S[wi * D::S + (size_t)i * DV + col0 + j] = sS[i * L::LS + j];
        }
        {   // U = U~ - W S to the workspace; sU holds diag(rk gamma_C / gamma) U (each thread its own elements)
            float acc[TU::NT][4];
            tile_zero(acc);
            mma_prod<TU::NT, DK, false, false>(acc, sW, L::LK, sS, L::LS, um, un, g, t);
            const float GC = sG[kC - 1];
#pragma unroll
            for (int q = 0; q < TU::NT; ++q)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = frow(um, g, e), j = fcol(un + q, t, e);
                    const float u = sU[r * L::LS + j] - acc[q][e];
                    sU[r * L::LS + j] = __expf(GC - sG[r]) * sRK[r] * u;
                    ws.U[wi * D::U + (size_t)r * DV + col0 + j] = u;
                }
        }
        __syncthreads();
        {   // S <- gamma_C S + K^T diag(gamma_C / gamma) U  (each thread updates its own elements)
            float acc[TS::NT][4];
            tile_zero(acc);
            mma_prod<TS::NT, kC, true, false, kEx, false>(acc, sK, L::LK, sU, L::LS, sm0, sn, g, t);
            const float gC = __expf(sG[kC - 1]);
#pragma unroll
            for (int q = 0; q < TS::NT; ++q)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float& s = sS[frow(sm0, g, e) * L::LS + fcol(sn + q, t, e)];
                    s = fmaf(gC, s, acc[q][e]);
                }
        }
        __syncthreads();
    }
    if (S_final) {   // the state after the last chunk (the forward's final state)
        for (int idx = tid; idx < DK * SW; idx += kStThreads) {
            const int i = idx / SW, j = idx % SW;
            S_final[sbase + (size_t)i * DV + j] = sS[i * L::LS + j];
        }
    }
}

// Adjoint chain, chunks in reverse: lam (= dL/dS at the chunk end) and dU to the workspace; dS0 at the end.
template <typename TT, int DK, int DV>
__global__ void __launch_bounds__(kStThreads)
bwd_state_adj_kernel(const TT* __restrict__ q, const TT* __restrict__ k, const TT* __restrict__ dout,
                     const float* __restrict__ dS_final, float* __restrict__ grad_S0, Ws ws, int T_len, int Hqk,
                     int Hv, const int32_t* __restrict__ cu, int nseq, float scale, bool vec) {
    using L = StSmem<DK, DV>;
    using D = WsDims<DK, DV>;
    constexpr int SW = L::SW, NSL = DV / SW;
    using TU = ChainTiles<kC, SW>;   // dU: C x SW
    using TS = ChainTiles<DK, SW>;   // lam: DK x SW
    constexpr bool kEx = sizeof(TT) == 2;   // bf16 K and dO are exact in tf32
    extern __shared__ __align__(16) float sm[];
    float* sW = sm + L::W_;
    float* sK = sm + L::K_;
    float* sQ = sm + L::Q_;
    float* sP = sm + L::P_;
    float* sdO = sm + L::X_;
    float* sdU = sm + L::Y_;
    float* sLam = sm + L::S_;
    float* sG = sm + L::G_;
    float* sQs = sm + L::R_;   // scale gamma_r
    const int sl = blockIdx.x % NSL, h = (blockIdx.x / NSL) % Hv, seq = blockIdx.x / (NSL * Hv);
    if (seq >= nseq) return;
    const int hk = h / (Hv / Hqk), col0 = sl * SW;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, g = lane / 4, t = lane % 4;
    const int um = 16 * (warp % TU::MT), un = (warp / TU::MT) * TU::NT;
    const int sm0 = 16 * (warp % TS::MT), sn = (warp / TS::MT) * TS::NT;
    long long t0, t1;
    seq_range(cu, seq, T_len, t0, t1);
    const long long nch = (t1 - t0 + kC - 1) / kC, slot0 = t0 / kC + seq;
    const size_t sbase = ((size_t)seq * Hv + h) * DK * DV + col0;
    for (int idx = tid; idx < DK * SW; idx += kStThreads) {
        const int i = idx / SW, j = idx % SW;
        sLam[i * L::LS + j] = dS_final ? dS_final[sbase + (size_t)i * DV + j] : 0.f;
    }
    for (long long c = nch - 1; c >= 0; --c) {
        const size_t wi = (size_t)(slot0 + c) * Hv + h;
        const long long tok0 = t0 + c * kC;
        const int n = (int)min((long long)kC, t1 - tok0);
        if (tid < kC) {
            const float gr = ws.G[wi * D::G + tid];
            sG[tid] = gr;
            sQs[tid] = scale * __expf(gr);
        }
        ld_ws<kC, DK, kStThreads>(sW, L::LK, ws.W + wi * D::W, DK, tid);
        ld_ws<kC, kC, kStThreads>(sP, L::LCC, ws.P + wi * D::P, kC, tid);
        ld_in<TT, kC, DK, kStThreads>(sK, L::LK, k + (tok0 * Hqk + hk) * DK, (size_t)Hqk * DK, n, tid, vec);
        ld_in<TT, kC, DK, kStThreads>(sQ, L::LK, q + (tok0 * Hqk + hk) * DK, (size_t)Hqk * DK, n, tid, vec);
        ld_in<TT, kC, SW, kStThreads>(sdO, L::LS, dout + (tok0 * Hv + h) * DV + col0, (size_t)Hv * DV, n, tid, vec);
        __syncthreads();
        for (int idx = tid; idx < DK * SW; idx += kStThreads) {
            const int i = idx / SW, j = idx % SW;
            ws.dS[wi * D::dS + (size_t)i * DV + col0 + j] = sLam[i * L::LS + j];
        }
        {   // dU = diag(gamma_C / gamma) K lam + P^T dO
            float kl[TU::NT][4], acc[TU::NT][4];
            tile_zero(kl);
            tile_zero(acc);
            mma_prod<TU::NT, DK, false, false, kEx, false>(kl, sK, L::LK, sLam, L::LS, um, un, g, t);
            mma_prod<TU::NT, kC, true, false, false, kEx>(acc, sP, L::LCC, sdO, L::LS, um, un, g, t);
            const float GC = sG[kC - 1];
#pragma unroll
            for (int qq = 0; qq < TU::NT; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = frow(um, g, e), j = fcol(un + qq, t, e);
                    const float du = fmaf(__expf(GC - sG[r]), kl[qq][e], acc[qq][e]);
                    sdU[r * L::LS + j] = du;
                    ws.dU[wi * D::dU + (size_t)r * DV + col0 + j] = du;
                }
        }
        __syncthreads();
        {   // lam <- gamma_C lam + Q^T diag(scale gamma) dO - W^T dU  (each thread updates its own elements)
            float acc[TS::NT][4], neg[TS::NT][4];
            tile_zero(acc);
            tile_zero(neg);
#pragma unroll 2
            for (int k0 = 0; k0 < kC; k0 += 8) {
                uint32_t ah[4], al[4];
                frag_at_scaled(sQ, L::LK, sQs, sm0, k0, g, t, ah, al);
#pragma unroll
                for (int qq = 0; qq < TS::NT; ++qq) {
                    uint32_t bh[2], bl[2];
                    frag_b<kEx>(sdO, L::LS, 8 * (sn + qq), k0, g, t, bh, bl);
                    mma_split<false, kEx>(acc[qq], ah, al, bh, bl);
                }
            }
            mma_prod<TS::NT, kC, true, false>(neg, sW, L::LK, sdU, L::LS, sm0, sn, g, t);
            const float gC = __expf(sG[kC - 1]);
#pragma unroll
            for (int qq = 0; qq < TS::NT; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float& l = sLam[frow(sm0, g, e) * L::LS + fcol(sn + qq, t, e)];
                    l = fmaf(gC, l, acc[qq][e] - neg[qq][e]);
                }
        }
        __syncthreads();
    }
    if (grad_S0) {
        for (int idx = tid; idx < DK * SW; idx += kStThreads) {
            const int i = idx / SW, j = idx % SW;
            grad_S0[sbase + (size_t)i * DV + j] = sLam[i * L::LS + j];
        }
    }
}

// ---------------------------------------------------------------- kernel 4: chunk-local gradients
// Every product runs on tf32 tensor cores with the three-product split (fp32 accuracy), in the
// accumulator fragment layout: warp w owns rows 16 (w % 4) .. +15 and, of a C x dk product, the
// n-tiles of 8 from (w / 4) dk / 32; of a C x C product, n-tiles 2 (w / 4) and 2 (w / 4) + 1.  dq and
// dk stay in those fragments across the value heads of the query/key head.
constexpr int kLoThreads = 512;   // 16 warps
constexpr int kDvc = 16;          // value columns per pass over dv (two buffer sets, the next pass loading)

__device__ __forceinline__ void cp_async16(float* smem, const float* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// fp32 workspace block rows [0, ROWS) x [0, WIDTH) to shared memory (leading dimension ld) by
// asynchronous 16-byte copies (both sides 16-byte aligned).
template <int ROWS, int WIDTH, int NT>
__device__ __forceinline__ void cp_ws(float* dst, int ld, const float* src, size_t stride, int tid) {
    constexpr int V = WIDTH / 4, TOTAL = ROWS * V;
    for (int idx = tid; idx < TOTAL; idx += NT) {
        const int r = idx / V, c = (idx % V) * 4;
        cp_async16(dst + r * ld + c, src + (size_t)r * stride + c);
    }
}

template <int DK, int DV>
struct LoSmem {
    // LK = 4 mod 32; LD = 20 (rows 20 banks apart: row-major fragment loads still hit 32 banks)
    static constexpr int LK = DK + 4, LD = kDvc + 4;
    static constexpr int K_ = 0, Q_ = K_ + kC * LK, KK_ = Q_ + kC * LK, QK_ = KK_ + kC * kLCC,
                         T_ = QK_ + kC * kLCC, X_ = T_ + kC * kLCC, DVB_ = X_ + kC * kLCC;
    // two sets of dv pass buffers (dU, U, dO, V: C x 16; S, lam: DK x 16), offsets within a set; afterwards
    // dW (C x DK) over them
    static constexpr int dU_ = 0, U_ = kC * LD, dO_ = 2 * kC * LD, V_ = 3 * kC * LD, S_ = 4 * kC * LD,
                         Lam_ = S_ + DK * LD, PS = Lam_ + DK * LD, DVB_END = DVB_ + 2 * PS, DW_END = DVB_ + kC * LK;
    static constexpr int VEC_ = DVB_END > DW_END ? DVB_END : DW_END;
    // G, beta, dG, dbeta, row scratch, h, the l2 scalars of K and Q rows, reduction scratch [8][C], warp sums
    static constexpr int G_ = VEC_, Beta_ = G_ + kC, dG_ = Beta_ + kC, dB_ = dG_ + kC, Row_ = dB_ + kC,
                         H_ = Row_ + kC, RK_ = H_ + kC, RQ_ = RK_ + kC, Scr_ = RQ_ + kC, Red_ = Scr_ + 8 * kC;
    static constexpr int FLOATS = Red_ + kLoThreads / 32;
    static constexpr size_t BYTES = (size_t)FLOATS * 4;
    static_assert(Q_ % 4 == 0 && KK_ % 4 == 0 && T_ % 4 == 0 && X_ % 4 == 0 && DVB_ % 4 == 0, "aligned regions");
};

// dst[r] += full sum of row r, given this thread's partial sums p0 (row row0 + g) and p1 (row row0 + g + 8):
// a quad sum over t, then the four column-group warps of the row tile in a fixed order.
__device__ __forceinline__ void frag_rows_add(float p0, float p1, float* scr, float* dst, int tid, int row0, int wg,
                                              int g, int t) {
    p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
    p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
    p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
    p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
    if (t == 0) {
        scr[wg * kC + row0 + g] = p0;
        scr[wg * kC + row0 + g + 8] = p1;
    }
    __syncthreads();
    if (tid < kC) dst[tid] += ((scr[tid] + scr[kC + tid]) + scr[2 * kC + tid]) + scr[3 * kC + tid];
    __syncthreads();
}

// dst[r] += rowsum_s F[r][s] - colsum_r F[r][s] for a C x C product in fragments (n-tiles 2 wg, 2 wg + 1):
// the derivative of sum F with respect to G through the ratios exp(G_r - G_s).
__device__ __forceinline__ void frag_rows_minus_cols(const float (&F)[2][4], float* scr, float* dst, int tid,
                                                     int row0, int wg, int mt, int g, int t) {
    float r0 = (F[0][0] + F[0][1]) + (F[1][0] + F[1][1]);
    float r1 = (F[0][2] + F[0][3]) + (F[1][2] + F[1][3]);
    r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
    r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
    float c[2][2];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float x = F[q][j] + F[q][2 + j];
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            c[q][j] = x;
        }
    if (t == 0) {
        scr[wg * kC + row0 + g] = r0;
        scr[wg * kC + row0 + g + 8] = r1;
    }
    if (g == 0) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int j = 0; j < 2; ++j) scr[(4 + mt) * kC + fcol(2 * wg + q, t, j)] = c[q][j];
    }
    __syncthreads();
    if (tid < kC) {
        const float rs = ((scr[tid] + scr[kC + tid]) + scr[2 * kC + tid]) + scr[3 * kC + tid];
        const float cs = ((scr[4 * kC + tid] + scr[5 * kC + tid]) + scr[6 * kC + tid]) + scr[7 * kC + tid];
        dst[tid] += rs - cs;
    }
    __syncthreads();
}

template <typename TT, int DK, int DV>
__global__ void __launch_bounds__(kLoThreads, 1)
bwd_local_kernel(const TT* __restrict__ q, const TT* __restrict__ k, const TT* __restrict__ v,
                 const TT* __restrict__ beta, const TT* __restrict__ dout, Ws ws, float* __restrict__ grad_q,
                 float* __restrict__ grad_k, float* __restrict__ grad_v, float* __restrict__ grad_g,
                 float* __restrict__ grad_beta, int T_len, int Hqk, int Hv, const int32_t* __restrict__ cu, int nseq,
                 float scale, bool vec, const float* __restrict__ A_log, const float* __restrict__ dt_bias,
                 bool normalize) {
    using L = LoSmem<DK, DV>;
    using D = WsDims<DK, DV>;
    constexpr int NTW = DK / 32;   // n-tiles of 8 per warp of a C x dk product
    constexpr bool kEx = sizeof(TT) == 2;   // bf16 inputs: K, Q, dO, V are exact in tf32
    extern __shared__ __align__(16) float sm[];
    float* sK = sm + L::K_;
    float* sQ = sm + L::Q_;
    float* sKK = sm + L::KK_;
    float* sQK = sm + L::QK_;
    float* sT = sm + L::T_;
    float* sX = sm + L::X_;
    float* sDW = sm + L::DVB_;
    float* sG = sm + L::G_;
    float* sBeta = sm + L::Beta_;
    float* sdG = sm + L::dG_;
    float* sdB = sm + L::dB_;
    float* sRow = sm + L::Row_;
    float* sH = sm + L::H_;
    float* sRK = sm + L::RK_;   // 1 / |k_r|, 1 / |q_r| with in-kernel normalisation, else 1
    float* sRQ = sm + L::RQ_;
    float* sScr = sm + L::Scr_;
    float* sRed = sm + L::Red_;

    const long long slot = blockIdx.x;
    const int hk = blockIdx.y, G = Hv / Hqk;
    int seq, n;
    long long tok0;
    if (!slot_chunk(cu, nseq, T_len, slot, seq, tok0, n)) return;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, g = lane / 4, t = lane % 4;
    const int mt = warp % 4, wg = warp / 4, row0 = 16 * mt, nb0 = wg * NTW, pb0 = 2 * wg;
    const int ra = row0 + g, rb = ra + 8;   // this thread's two accumulator rows

    ld_in<TT, kC, DK, kLoThreads>(sK, L::LK, k + (tok0 * Hqk + hk) * DK, (size_t)Hqk * DK, n, tid, vec);
    ld_in<TT, kC, DK, kLoThreads>(sQ, L::LK, q + (tok0 * Hqk + hk) * DK, (size_t)Hqk * DK, n, tid, vec);
    if (tid < kC) {   // the WY kernel's l2 scalars (the same for every value head of this query/key head)
        const size_t w0 = (size_t)slot * Hv + (size_t)hk * G;
        sRK[tid] = normalize ? ws.R[w0 * D::R + tid] : 1.f;
        sRQ[tid] = normalize ? ws.R[w0 * D::R + kC + tid] : 1.f;
    }
    __syncthreads();
    // K and Q stay as loaded (exact for bf16 inputs); the normalised rows diag(rk) K and diag(rq) Q enter
    // through the scalars: on the Gram entries, on the A columns of the products with K or Q as B, and on
    // the row sums and the products' columns below.
    {   // Gram matrices K_n K_n^T and Q_n K_n^T (shared by the value heads)
        float kk[2][4], qk[2][4];
        tile_zero(kk);
        tile_zero(qk);
        mma_prod<2, DK, false, true, kEx, kEx>(kk, sK, L::LK, sK, L::LK, row0, pb0, g, t);
        mma_prod<2, DK, false, true, kEx, kEx>(qk, sQ, L::LK, sK, L::LK, row0, pb0, g, t);
        if (normalize) {
#pragma unroll
            for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = frow(row0, g, e), c = fcol(pb0 + qq, t, e);
                    kk[qq][e] *= sRK[r] * sRK[c];
                    qk[qq][e] *= sRQ[r] * sRK[c];
                }
        }
        store_frag<2>(sKK, kLCC, kk, row0, pb0, g, t, 1.f);
        store_frag<2>(sQK, kLCC, qk, row0, pb0, g, t, 1.f);
    }

    for (int jh = 0; jh < G; ++jh) {
        const int h = hk * G + jh;
        const size_t wi = (size_t)slot * Hv + h;
        ld_ws<kC, kC, kLoThreads>(sT, kLCC, ws.T + wi * D::T, kC, tid);
        if (tid < kC) {
            sG[tid] = ws.G[wi * D::G + tid];
            float bt = tid < n ? to_f32(beta[(tok0 + tid) * Hv + h]) : 0.f;
            if (A_log && tid < n) {   // beta from the raw projection b, as the WY kernel forms it
                float gt;
                gates_from_raw(0.f, bt, A_log[h], dt_bias[h], gt, bt);
            }
            sBeta[tid] = bt;
            sdG[tid] = 0.f;
            sdB[tid] = 0.f;
            sH[tid] = 0.f;
        }
        // fW: dU S^T, fX: dO S^T, fY: U lam^T (n-tiles from nb0); fP: dO U^T, fTv: dU V^T (n-tiles from pb0)
        float fW[NTW][4], fX[NTW][4], fY[NTW][4], fP[2][4], fTv[2][4];
        tile_zero(fW);
        tile_zero(fX);
        tile_zero(fY);
        tile_zero(fP);
        tile_zero(fTv);
        float zv0 = 0.f, zv1 = 0.f, ss = 0.f;
        // Passes over dv, double-buffered: while pass p computes, the fp32 workspace blocks of pass p + 1
        // arrive by cp.async in the other buffer set and its dO / V rows (16-byte pieces, one per thread)
        // wait in registers.
        constexpr int NP = DV / kDvc;
        constexpr int EPV = 16 / (int)sizeof(TT), PPR = kDvc / EPV, PIECES = kC * PPR;   // per dO or V block
        static_assert(2 * PIECES <= kLoThreads, "one input piece per thread");
        const TT* in_base[2] = {dout + (tok0 * Hv + h) * DV, v + (tok0 * Hv + h) * DV};
        const int pw = tid / PIECES, pr = (tid % PIECES) / PPR, pc = (tid % PIECES) % PPR * EPV;
        uint4 piece = make_uint4(0u, 0u, 0u, 0u);
        auto issue_pass = [&](int p) {   // fp32 blocks of pass p into set p & 1; its dO / V piece into registers
            float* B = sm + L::DVB_ + (p & 1) * L::PS;
            const int jc = p * kDvc;
            cp_ws<kC, kDvc, kLoThreads>(B + L::dU_, L::LD, ws.dU + wi * D::dU + jc, DV, tid);
            cp_ws<kC, kDvc, kLoThreads>(B + L::U_, L::LD, ws.U + wi * D::U + jc, DV, tid);
            cp_ws<DK, kDvc, kLoThreads>(B + L::S_, L::LD, ws.S + wi * D::S + jc, DV, tid);
            cp_ws<DK, kDvc, kLoThreads>(B + L::Lam_, L::LD, ws.dS + wi * D::dS + jc, DV, tid);
            cp_async_commit();
            piece = make_uint4(0u, 0u, 0u, 0u);
            if (vec && pw < 2 && pr < n)
                piece = *reinterpret_cast<const uint4*>(in_base[pw] + (size_t)pr * Hv * DV + jc + pc);
        };
        issue_pass(0);
        for (int p = 0; p < NP; ++p) {
            const int jc = p * kDvc;
            float* B = sm + L::DVB_ + (p & 1) * L::PS;
            float* sdU = B + L::dU_;
            float* sU = B + L::U_;
            float* sdO = B + L::dO_;
            float* sV = B + L::V_;
            float* sS = B + L::S_;
            float* sLam = B + L::Lam_;
            if (vec) {   // this pass's dO / V piece, converted to fp32
                if (pw < 2) {
                    float f[EPV];
                    unpack16(piece, f);
                    float* d = (pw == 0 ? sdO : sV) + pr * L::LD + pc;
#pragma unroll
                    for (int x = 0; x < EPV; ++x) d[x] = f[x];
                }
            } else {
                ld_in<TT, kC, kDvc, kLoThreads>(sdO, L::LD, in_base[0] + jc, (size_t)Hv * DV, n, tid, false);
                ld_in<TT, kC, kDvc, kLoThreads>(sV, L::LD, in_base[1] + jc, (size_t)Hv * DV, n, tid, false);
            }
            if (p + 1 < NP) {
                issue_pass(p + 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            for (int idx = tid; idx < DK * kDvc; idx += kLoThreads) {
                const int i = idx / kDvc, j = idx % kDvc;
                ss = fmaf(sS[i * L::LD + j], sLam[i * L::LD + j], ss);
            }
#pragma unroll
            for (int k0 = 0; k0 < kDvc; k0 += 8) {   // dU S^T, dU V^T, dO S^T, dO U^T, U lam^T
                uint32_t ah[4], al[4], bh[2], bl[2], sh[NTW][2], sl[NTW][2];
#pragma unroll
                for (int qq = 0; qq < NTW; ++qq) frag_bt(sS, L::LD, 8 * (nb0 + qq), k0, g, t, sh[qq], sl[qq]);
                frag_a(sdU, L::LD, row0, k0, g, t, ah, al);
#pragma unroll
                for (int qq = 0; qq < NTW; ++qq) mma_3xtf32(fW[qq], ah, al, sh[qq], sl[qq]);
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    frag_bt<kEx>(sV, L::LD, 8 * (pb0 + qq), k0, g, t, bh, bl);
                    mma_split<false, kEx>(fTv[qq], ah, al, bh, bl);
                }
                frag_a<kEx>(sdO, L::LD, row0, k0, g, t, ah, al);
#pragma unroll
                for (int qq = 0; qq < NTW; ++qq) mma_split<kEx, false>(fX[qq], ah, al, sh[qq], sl[qq]);
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    frag_bt(sU, L::LD, 8 * (pb0 + qq), k0, g, t, bh, bl);
                    mma_split<kEx, false>(fP[qq], ah, al, bh, bl);
                }
#pragma unroll
                for (int qq = 0; qq < NTW; ++qq) frag_bt(sLam, L::LD, 8 * (nb0 + qq), k0, g, t, sh[qq], sl[qq]);
                frag_a(sU, L::LD, row0, k0, g, t, ah, al);
#pragma unroll
                for (int qq = 0; qq < NTW; ++qq) mma_3xtf32(fY[qq], ah, al, sh[qq], sl[qq]);
            }
            if (wg < kDvc / 8) {   // dV = diag(beta) T^T dU (columns 8 wg .. 8 wg + 7);  dbeta += rowsum(T^T dU o V)
                float z[1][4];
                tile_zero(z);
                mma_prod<1, kC, true, false>(z, sT, kLCC, sdU, L::LD, row0, wg, g, t);
                const int j = fcol(wg, t, 0);
                zv0 = fmaf(z[0][0], sV[ra * L::LD + j], fmaf(z[0][1], sV[ra * L::LD + j + 1], zv0));
                zv1 = fmaf(z[0][2], sV[rb * L::LD + j], fmaf(z[0][3], sV[rb * L::LD + j + 1], zv1));
                if (ra < n) {   // (grad_v needs only 4-byte alignment: scalar stores)
                    float* o = grad_v + ((tok0 + ra) * Hv + h) * DV + jc + j;
                    o[0] = sBeta[ra] * z[0][0];
                    o[1] = sBeta[ra] * z[0][1];
                }
                if (rb < n) {
                    float* o = grad_v + ((tok0 + rb) * Hv + h) * DV + jc + j;
                    o[0] = sBeta[rb] * z[0][2];
                    o[1] = sBeta[rb] * z[0][3];
                }
            }
            __syncthreads();   // this set is free for pass p + 2
        }
        {   // gamma_C <lam, S>: warp sums of ss (added below)
            float x = ss;
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
            if (lane == 0) sRed[warp] = x;
        }
        frag_rows_add(zv0, zv1, sScr, sdB, tid, row0, wg, g, t);
        store_frag<NTW>(sDW, L::LK, fW, row0, nb0, g, t, -1.f);      // dW = -dU S^T (over the pass buffers)
        // dQ = scale diag(gamma) (dO S^T) in fX;  dG_r += scale gamma_r (dO S^T)_r . q_r
        // dK = diag(gamma_C / gamma) (U lam^T) in fY;  with h_r = (gamma_C / gamma_r) (U lam^T)_r . k_r:
        // dG_r -= h_r and dG_{C-1} += sum_r h_r + gamma_C <lam, S>
        float (&dQ)[NTW][4] = fX;
        float (&dK)[NTW][4] = fY;
        const float GC = sG[kC - 1];
        {
            const float gra = scale * __expf(sG[ra]), grb = scale * __expf(sG[rb]);
            const float kca = __expf(GC - sG[ra]), kcb = __expf(GC - sG[rb]);
            float xa = 0.f, xb = 0.f, ya = 0.f, yb = 0.f;
#pragma unroll
            for (int qq = 0; qq < NTW; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = frow(row0, g, e), c = fcol(nb0 + qq, t, e);
                    const float xq = fX[qq][e] * sQ[r * L::LK + c], yk = fY[qq][e] * sK[r * L::LK + c];
                    if (e < 2) { xa += xq; ya += yk; } else { xb += xq; yb += yk; }
                    dQ[qq][e] = (e < 2 ? gra : grb) * fX[qq][e];
                    dK[qq][e] = (e < 2 ? kca : kcb) * fY[qq][e];
                }
            frag_rows_add(gra * sRQ[ra] * xa, grb * sRQ[rb] * xb, sScr, sdG, tid, row0, wg, g, t);
            frag_rows_add(-kca * sRK[ra] * ya, -kcb * sRK[rb] * yb, sScr, sH, tid, row0, wg, g, t);   // sH = -h
        }
        if (tid < 32) {
            float th = sH[tid] + sH[tid + 32], tl = tid < kLoThreads / 32 ? sRed[tid] : 0.f;
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) {
                th += __shfl_xor_sync(0xffffffffu, th, m);
                tl += __shfl_xor_sync(0xffffffffu, tl, m);
            }
            if (tid == 0) sdG[kC - 1] += __expf(GC) * tl - th;
        }
        __syncthreads();
        if (tid < kC) sdG[tid] += sH[tid];
        {   // E = scale D o dP (s <= r) -> sX (row-major);  dG from E o QK^T
            float F[2][4];
#pragma unroll
            for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = frow(row0, g, e), s = fcol(pb0 + qq, t, e);
                    const float ev = s <= r ? scale * __expf(sG[r] - sG[s]) * fP[qq][e] : 0.f;
                    sX[r * kLCC + s] = ev;
                    F[qq][e] = ev * sQK[r * kLCC + s];
                }
            frag_rows_minus_cols(F, sScr, sdG, tid, row0, wg, mt, g, t);   // its barriers publish sX and sDW
        }
        mma_prod_as<NTW, kC, false, kEx>(dQ, sX, kLCC, sRK, sK, L::LK, row0, nb0, g, t);   // dQ += E diag(rk) K
        mma_prod_as<NTW, kC, true, kEx>(dK, sX, kLCC, sRQ, sQ, L::LK, row0, nb0, g, t);    // dK += E^T diag(rq) Q
        {   // R = T^T dW;  dK += diag(beta gamma) R;  dbeta_s += gamma_s R_s.k_s;  dG_s += beta_s gamma_s R_s.k_s
            float R[NTW][4];
            tile_zero(R);
            mma_prod<NTW, kC, true, false>(R, sT, kLCC, sDW, L::LK, row0, nb0, g, t);
            const float gma = __expf(sG[ra]), gmb = __expf(sG[rb]);
            const float bga = sBeta[ra] * gma, bgb = sBeta[rb] * gmb;
            float rka = 0.f, rkb = 0.f;
#pragma unroll
            for (int qq = 0; qq < NTW; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = frow(row0, g, e), c = fcol(nb0 + qq, t, e);
                    const float x = R[qq][e] * sK[r * L::LK + c];
                    if (e < 2) rka += x; else rkb += x;
                    dK[qq][e] = fmaf(e < 2 ? bga : bgb, R[qq][e], dK[qq][e]);
                }
            rka *= sRK[ra];
            rkb *= sRK[rb];
            frag_rows_add(gma * rka, gmb * rkb, sScr, sdB, tid, row0, wg, g, t);   // also ends the reads of E
            frag_rows_add(bga * rka, bgb * rkb, sScr, sdG, tid, row0, wg, g, t);
        }
        {   // dT = (dU V^T + dW K^T diag(gamma)) diag(beta), lower part -> sX
            float Tk[2][4];
            tile_zero(Tk);
            mma_prod<2, DK, false, true, false, kEx>(Tk, sDW, L::LK, sK, L::LK, row0, pb0, g, t);
#pragma unroll
            for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = frow(row0, g, e), s = fcol(pb0 + qq, t, e);
                    sX[r * kLCC + s] = s <= r ? sBeta[s] * fmaf(__expf(sG[s]) * sRK[s], Tk[qq][e], fTv[qq][e]) : 0.f;
                }
        }
        __syncthreads();
        {   // M1 = T^T dT -> sX
            float M1[2][4];
            tile_zero(M1);
            mma_prod<2, kC, true, false>(M1, sT, kLCC, sX, kLCC, row0, pb0, g, t);
            __syncthreads();
            store_frag<2>(sX, kLCC, M1, row0, pb0, g, t, 1.f);
        }
        __syncthreads();
        {   // dM = -(M1 T^T) strictly lower;  dbeta_r += sum_s dM_rs A_rs;  H = diag(beta) D o dM, and
            // sX <- H + H^T (symmetric, so one product gives H K + H^T K)
            float Mm[2][4];
            tile_zero(Mm);
            mma_prod<2, kC, false, true>(Mm, sX, kLCC, sT, kLCC, row0, pb0, g, t);
            float F[2][4], ba = 0.f, bb = 0.f;
            __syncthreads();
#pragma unroll
            for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = frow(row0, g, e), s = fcol(pb0 + qq, t, e);
                    float f = 0.f;
                    if (s < r) {
                        const float d = __expf(sG[r] - sG[s]), kk = sKK[r * kLCC + s], dm = -Mm[qq][e];
                        const float hv = sBeta[r] * d * dm;
                        if (e < 2) ba = fmaf(dm, d * kk, ba); else bb = fmaf(dm, d * kk, bb);
                        f = hv * kk;
                        sX[r * kLCC + s] = hv;
                        sX[s * kLCC + r] = hv;
                    } else if (s == r) {
                        sX[r * kLCC + s] = 0.f;
                    }
                    F[qq][e] = f;
                }
            frag_rows_add(ba, bb, sScr, sdB, tid, row0, wg, g, t);
            frag_rows_minus_cols(F, sScr, sdG, tid, row0, wg, mt, g, t);
        }
        mma_prod_as<NTW, kC, false, kEx>(dK, sX, kLCC, sRK, sK, L::LK, row0, nb0, g, t);   // dK += (H + H^T) diag(rk) K
        if (tid < 32) {   // dg = suffix sums of dG: lane l holds tokens 2l, 2l + 1
            const float a = sdG[2 * tid], b = sdG[2 * tid + 1];
            float x = a + b;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, x, o);
                if (tid + o < 32) x += y;
            }
            sRow[2 * tid] = x;
            sRow[2 * tid + 1] = x - a;
        }
        __syncthreads();
        if (tid < n) {
            grad_g[(tok0 + tid) * Hv + h] = sRow[tid];
            grad_beta[(tok0 + tid) * Hv + h] = sdB[tid];
        }
        // dq, dk of the query/key head: its first value head writes, the others add (same thread, same element)
#pragma unroll
        for (int qq = 0; qq < NTW; ++qq)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = frow(row0, g, e);
                if (r < n) {
                    const size_t o = ((tok0 + r) * Hqk + hk) * DK + fcol(nb0 + qq, t, e);
                    grad_q[o] = jh == 0 ? dQ[qq][e] : grad_q[o] + dQ[qq][e];
                    grad_k[o] = jh == 0 ? dK[qq][e] : grad_k[o] + dK[qq][e];
                }
            }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- chunked forward (any head dims, fp32 accuracy)
// The prefill through the same chunk algebra: the WY kernel, the forward chain (chunk-start states,
// U, and the final state), then per chunk O = scale diag(gamma) Q S + P U with P = scale D o (Q K^T)
// (s <= r), which is the unrolled read o_r = scale S_r^T q_r.
template <int DK, int DV>
struct OutSmem {
    static constexpr int LK = DK + 4, LV = DV + 4;
    static constexpr int Q_ = 0, S_ = Q_ + kC * LK, P_ = S_ + DK * LV, U_ = P_ + kC * kLCC, G_ = U_ + kC * LV,
                         R_ = G_ + kC;
    static constexpr int FLOATS = R_ + kC;
    static constexpr size_t BYTES = (size_t)FLOATS * 4;
    static_assert(S_ % 4 == 0 && P_ % 4 == 0 && U_ % 4 == 0, "16-byte aligned regions");
};

template <typename TT, int DK, int DV>
__global__ void __launch_bounds__(kStThreads)
fwd_out_kernel(const TT* __restrict__ q, TT* __restrict__ out, Ws ws, int T_len, int Hqk, int Hv,
               const int32_t* __restrict__ cu, int nseq, float scale, bool vec, bool normalize) {
    using L = OutSmem<DK, DV>;
    using D = WsDims<DK, DV>;
    using TO = ChainTiles<kC, DV>;
    constexpr bool kEx = sizeof(TT) == 2;   // bf16 Q is exact in tf32
    extern __shared__ __align__(16) float sm[];
    float* sQ = sm + L::Q_;
    float* sS = sm + L::S_;
    float* sP = sm + L::P_;
    float* sU = sm + L::U_;
    float* sG = sm + L::G_;
    float* sRQ = sm + L::R_;   // per-row l2 scalars of Q (P already carries them)
    const long long slot = blockIdx.x;
    const int hk = blockIdx.y, G = Hv / Hqk;
    int seq, n;
    long long tok0;
    if (!slot_chunk(cu, nseq, T_len, slot, seq, tok0, n)) return;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, g = lane / 4, t = lane % 4;
    const int om = 16 * (warp % TO::MT), on = (warp / TO::MT) * TO::NT;
    ld_in<TT, kC, DK, kStThreads>(sQ, L::LK, q + (tok0 * Hqk + hk) * DK, (size_t)Hqk * DK, n, tid, vec);
    for (int jh = 0; jh < G; ++jh) {
        const int h = hk * G + jh;
        const size_t wi = (size_t)slot * Hv + h;
        if (tid < kC) {
            sG[tid] = ws.G[wi * D::G + tid];
            sRQ[tid] = normalize ? ws.R[wi * D::R + kC + tid] : 1.f;
        }
        ld_ws<DK, DV, kStThreads>(sS, L::LV, ws.S + wi * D::S, DV, tid);
        ld_ws<kC, kC, kStThreads>(sP, kLCC, ws.P + wi * D::P, kC, tid);
        ld_ws<kC, DV, kStThreads>(sU, L::LV, ws.U + wi * D::U, DV, tid);
        __syncthreads();
        float y1[TO::NT][4], y2[TO::NT][4];
        tile_zero(y1);
        tile_zero(y2);
        mma_prod<TO::NT, DK, false, false, kEx, false>(y1, sQ, L::LK, sS, L::LV, om, on, g, t);   // Q S
        mma_prod<TO::NT, kC, false, false>(y2, sP, kLCC, sU, L::LV, om, on, g, t);              // P U
        const int ra = om + g, rb = ra + 8;
        const float ca = scale * __expf(sG[ra]) * sRQ[ra], cb = scale * __expf(sG[rb]) * sRQ[rb];
#pragma unroll
        for (int qq = 0; qq < TO::NT; ++qq) {
            const int j = fcol(on + qq, t, 0);
            if (ra < n) {
                TT* o = out + ((tok0 + ra) * Hv + h) * DV + j;
                o[0] = from_f32<TT>(fmaf(ca, y1[qq][0], y2[qq][0]));
                o[1] = from_f32<TT>(fmaf(ca, y1[qq][1], y2[qq][1]));
            }
            if (rb < n) {
                TT* o = out + ((tok0 + rb) * Hv + h) * DV + j;
                o[0] = from_f32<TT>(fmaf(cb, y1[qq][2], y2[qq][2]));
                o[1] = from_f32<TT>(fmaf(cb, y1[qq][3], y2[qq][3]));
            }
        }
        __syncthreads();
    }
}

template <typename TT, int DK, int DV>
cudaError_t launch_fwd_typed(const PrefillArgs& a, const BwdLayout& Lw) {
    uint8_t* base = static_cast<uint8_t*>(a.workspace);
    Ws ws{};
    ws.T = reinterpret_cast<float*>(base + Lw.T_off);
    ws.P = reinterpret_cast<float*>(base + Lw.P_off);
    ws.W = reinterpret_cast<float*>(base + Lw.W_off);
    ws.U = reinterpret_cast<float*>(base + Lw.U_off);
    ws.G = reinterpret_cast<float*>(base + Lw.G_off);
    ws.S = reinterpret_cast<float*>(base + Lw.S_off);
    ws.R = reinterpret_cast<float*>(base + Lw.R_off);
    const TT* q = static_cast<const TT*>(a.q);
    const TT* k = static_cast<const TT*>(a.k);
    const TT* v = static_cast<const TT*>(a.v);
    const TT* g = static_cast<const TT*>(a.g);
    const TT* beta = static_cast<const TT*>(a.beta);
    TT* out = static_cast<TT*>(a.out);
    constexpr int NSL = DV / slice_width<DV>();
    // the prefill entry point requires 16-byte aligned q, k, v and out
    const bool vec = true;
    using S1 = WySmem<DK, DV>;
    using S2 = StSmem<DK, DV>;
    using S3 = OutSmem<DK, DV>;
    cudaError_t e;
    if ((e = set_smem2(bwd_wy_kernel<TT, DK, DV>, S1::BYTES)) != cudaSuccess) return e;
    if ((e = set_smem(bwd_state_fwd_kernel<TT, DK, DV>, S2::BYTES)) != cudaSuccess) return e;
    if ((e = set_smem(fwd_out_kernel<TT, DK, DV>, S3::BYTES)) != cudaSuccess) return e;
    const dim3 chunk_grid((unsigned)Lw.slots, (unsigned)a.Hqk);
    const unsigned nst = (unsigned)((long long)a.num_seqs * a.Hv * NSL);
    const bool normalize = (a.flags & GDN_NORMALIZE_QK) != 0;
    const float* A_log = (a.flags & GDN_RAW_GATES) ? a.A_log : nullptr;
    bwd_wy_kernel<TT, DK, DV><<<chunk_grid, kWyThreads, S1::BYTES, a.stream>>>(
        q, k, v, g, beta, ws, a.T, a.Hqk, a.Hv, a.cu_seqlens, a.num_seqs, a.scale, vec, A_log, a.dt_bias, normalize);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_state_fwd_kernel<TT, DK, DV><<<nst, kStThreads, S2::BYTES, a.stream>>>(
        k, a.S0, a.S_final, ws, a.T, a.Hqk, a.Hv, a.cu_seqlens, a.num_seqs, vec, normalize);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fwd_out_kernel<TT, DK, DV><<<chunk_grid, kStThreads, S3::BYTES, a.stream>>>(
        q, out, ws, a.T, a.Hqk, a.Hv, a.cu_seqlens, a.num_seqs, a.scale, vec, normalize);
    return cudaGetLastError();
}

template <typename TT, int DK>
cudaError_t launch_fwd_dk(const PrefillArgs& a, const BwdLayout& L) {
    switch (a.dv) {
        case 32: return launch_fwd_typed<TT, DK, 32>(a, L);
        case 64: return launch_fwd_typed<TT, DK, 64>(a, L);
        case 128: return launch_fwd_typed<TT, DK, 128>(a, L);
    }
    return cudaErrorInvalidValue;
}

template <typename TT>
cudaError_t launch_fwd_dtype(const PrefillArgs& a, const BwdLayout& L) {
    switch (a.dk) {
        case 32: return launch_fwd_dk<TT, 32>(a, L);
        case 64: return launch_fwd_dk<TT, 64>(a, L);
        case 128: return launch_fwd_dk<TT, 128>(a, L);
    }
    return cudaErrorInvalidValue;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <typename F>
cudaError_t set_smem(F* kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
// The same, with the largest shared-memory carveout: for kernels that run two CTAs per SM.
template <typename F>
cudaError_t set_smem2(F* kernel, size_t bytes) {
    const cudaError_t e = set_smem(kernel, bytes);
    return e == cudaSuccess ? cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) : e;
}

template <typename TT, int DK, int DV>
cudaError_t launch_typed(const BackwardArgs& a, const BwdLayout& Lw) {
    uint8_t* base = static_cast<uint8_t*>(a.workspace);
    Ws ws{};
    ws.T = reinterpret_cast<float*>(base + Lw.T_off);
    ws.P = reinterpret_cast<float*>(base + Lw.P_off);
    ws.W = reinterpret_cast<float*>(base + Lw.W_off);
    ws.U = reinterpret_cast<float*>(base + Lw.U_off);
    ws.G = reinterpret_cast<float*>(base + Lw.G_off);
    ws.S = reinterpret_cast<float*>(base + Lw.S_off);
    ws.dS = reinterpret_cast<float*>(base + Lw.dS_off);
    ws.dU = reinterpret_cast<float*>(base + Lw.dU_off);
    const bool front_end = (a.flags & (GDN_NORMALIZE_QK | GDN_RAW_GATES)) != 0;
    ws.R = front_end ? reinterpret_cast<float*>(base + Lw.R_off) : nullptr;
    const TT* q = static_cast<const TT*>(a.q);
    const TT* k = static_cast<const TT*>(a.k);
    const TT* v = static_cast<const TT*>(a.v);
    const TT* g = static_cast<const TT*>(a.g);
    const TT* beta = static_cast<const TT*>(a.beta);
    const TT* dout = static_cast<const TT*>(a.dout);
    constexpr int NSL = DV / slice_width<DV>();
    cudaError_t e;
    const auto mark = [&](int i) {
        if (a.events && i < a.num_events && a.events[i]) cudaEventRecord(static_cast<cudaEvent_t>(a.events[i]), a.stream);
    };
    // 16-byte vector loads of the inputs need 16-byte aligned bases (row strides are multiples of 16 bytes)
    const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool vec = al16(a.q) && al16(a.k) && al16(a.v) && al16(a.dout);

    using S1 = WySmem<DK, DV>;
    using S2 = StSmem<DK, DV>;
    using S4 = LoSmem<DK, DV>;
    const dim3 chunk_grid((unsigned)Lw.slots, (unsigned)a.Hqk);
    const unsigned nst = (unsigned)((long long)a.num_seqs * a.Hv * NSL);
    if ((e = set_smem2(bwd_wy_kernel<TT, DK, DV>, S1::BYTES)) != cudaSuccess) return e;
    if ((e = set_smem(bwd_state_fwd_kernel<TT, DK, DV>, S2::BYTES)) != cudaSuccess) return e;
    if ((e = set_smem(bwd_state_adj_kernel<TT, DK, DV>, S2::BYTES)) != cudaSuccess) return e;
    if ((e = set_smem(bwd_local_kernel<TT, DK, DV>, S4::BYTES)) != cudaSuccess) return e;

    // With the front end (only for bf16, dk = dv = 128: the caller checks), every kernel takes the raw inputs
    // with the l2 scalars and the gates inside (the WY kernel forms them and keeps the scalars per chunk).
    const bool normalize = (a.flags & GDN_NORMALIZE_QK) != 0;
    const float* A_log = (a.flags & GDN_RAW_GATES) ? a.A_log : nullptr;
    bwd_wy_kernel<TT, DK, DV><<<chunk_grid, kWyThreads, S1::BYTES, a.stream>>>(
        q, k, v, g, beta, ws, a.T, a.Hqk, a.Hv, a.cu_seqlens, a.num_seqs, a.scale, vec, A_log, a.dt_bias, normalize);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark(1);
    // the forward chain: on the tcgen05 tensor cores for bf16 inputs with dk = dv = 128 (16-byte aligned k)
    e = cudaErrorNotSupported;
    if constexpr (sizeof(TT) == 2 && DK == 128 && DV == 128)
        e = launch_bwd_state_fwd_tc(a.k, a.S0, nullptr, ws.W, ws.U, ws.G, ws.S, normalize ? ws.R : nullptr, a.T, a.Hqk,
                                    a.Hv, a.cu_seqlens, a.num_seqs, normalize, a.stream, a.status);
    if (e == cudaErrorNotSupported)
        bwd_state_fwd_kernel<TT, DK, DV><<<nst, kStThreads, S2::BYTES, a.stream>>>(
            k, a.S0, nullptr, ws, a.T, a.Hqk, a.Hv, a.cu_seqlens, a.num_seqs, vec, normalize);
    else if (e != cudaSuccess)
        return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark(2);
    // the adjoint chain: on the tcgen05 tensor cores for bf16 inputs with dk = dv = 128 (16-byte aligned q, k, dout)
    e = cudaErrorNotSupported;
    if constexpr (sizeof(TT) == 2 && DK == 128 && DV == 128)
        e = launch_bwd_state_adj_tc(a.q, a.k, a.dout, a.dS_final, a.grad_S0, ws.W, ws.P, ws.G, ws.dS, ws.dU, a.T, a.Hqk,
                                    a.Hv, a.cu_seqlens, a.num_seqs, a.scale, a.stream, a.status,
                                    normalize ? ws.R : nullptr, normalize);
    if (e == cudaErrorNotSupported && front_end) return e;   // the general adjoint chain has no front end
    if (e == cudaErrorNotSupported)
        bwd_state_adj_kernel<TT, DK, DV><<<nst, kStThreads, S2::BYTES, a.stream>>>(
            q, k, dout, a.dS_final, a.grad_S0, ws, a.T, a.Hqk, a.Hv, a.cu_seqlens, a.num_seqs, a.scale, vec);
    else if (e != cudaSuccess)
        return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark(3);
    // with the front end, on the raw rows as well: the WY kernel's l2 scalars, beta from the raw b
    bwd_local_kernel<TT, DK, DV><<<chunk_grid, kLoThreads, S4::BYTES, a.stream>>>(
        q, k, v, beta, dout, ws, a.grad_q, a.grad_k, a.grad_v, a.grad_g, a.grad_beta, a.T, a.Hqk, a.Hv,
        a.cu_seqlens, a.num_seqs, a.scale, vec, A_log, a.dt_bias, normalize);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark(4);
    return cudaSuccess;
}

template <typename TT, int DK>
cudaError_t launch_dk(const BackwardArgs& a, const BwdLayout& L) {
    switch (a.dv) {
        case 32: return launch_typed<TT, DK, 32>(a, L);
        case 64: return launch_typed<TT, DK, 64>(a, L);
        case 128: return launch_typed<TT, DK, 128>(a, L);
    }
    return cudaErrorInvalidValue;
}

template <typename TT>
cudaError_t launch_dtype(const BackwardArgs& a, const BwdLayout& L) {
    switch (a.dk) {
        case 32: return launch_dk<TT, 32>(a, L);
        case 64: return launch_dk<TT, 64>(a, L);
        case 128: return launch_dk<TT, 128>(a, L);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

BwdLayout backward_layout(int B, int T, int Hv, int dk, int dv, int nseq, bool packed, bool adjoint, bool with_r) {
    const long long ttot = packed ? (long long)T : (long long)B * T;
    BwdLayout L{};
    L.slots = (ttot + kC - 1) / kC + nseq;
    const size_t per = (size_t)L.slots * Hv * sizeof(float);
    size_t off = 0;
    const auto take = [&](size_t& field, size_t floats) {
        field = off;
        off = align256(off + per * floats);
    };
    take(L.T_off, (size_t)kC * kC);
    take(L.P_off, (size_t)kC * kC);
    take(L.W_off, (size_t)kC * dk);
    take(L.U_off, (size_t)kC * dv);
    take(L.G_off, (size_t)kC);
    take(L.S_off, (size_t)dk * dv);
    if (adjoint) {
        take(L.dS_off, (size_t)dk * dv);
        take(L.dU_off, (size_t)kC * dv);
        if (with_r) take(L.R_off, (size_t)2 * kC);   // the front end's per-row l2 scalars
    } else {
        take(L.R_off, (size_t)2 * kC);   // the prefill front end's per-row l2 scalars
    }
    L.total = off;
    return L;
}

size_t chunked_prefill_workspace_bytes(int B, int T, int Hv, int dk, int dv, int nseq, bool packed) {
    return backward_layout(B, T, Hv, dk, dv, nseq, packed, false).total;
}

cudaError_t launch_chunked_prefill(const PrefillArgs& a) {
    const BwdLayout L = backward_layout(a.B, a.T, a.Hv, a.dk, a.dv, a.num_seqs, a.cu_seqlens != nullptr, false);
    return a.dtype == GDN_BF16 ? launch_fwd_dtype<__nv_bfloat16>(a, L) : launch_fwd_dtype<float>(a, L);
}

cudaError_t launch_backward(const BackwardArgs& a) {
    const bool front_end = (a.flags & (GDN_NORMALIZE_QK | GDN_RAW_GATES)) != 0;
    const BwdLayout L = backward_layout(a.B, a.T, a.Hv, a.dk, a.dv, a.num_seqs, a.cu_seqlens != nullptr, true, front_end);
    return a.dtype == GDN_BF16 ? launch_dtype<__nv_bfloat16>(a, L) : launch_dtype<float>(a, L);
}

}  // namespace gdn
