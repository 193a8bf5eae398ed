// Chunk-parallel prefill on the sm_103a tensor cores (tcgen05.mma kind::f16, bf16 operands, fp32
// accumulators in TMEM, operands staged in shared memory by TMA / bulk copies).
//
// The chunk algebra follows from the update of "Transformer by Hand, ch. 7", section "The formula"
// (the learn-llm "linear attention" page notes that the chunked implementations are mathematically
// equivalent to the token loop).  Inside a chunk of C = 64 tokens of one (sequence, value head), with
// G_r = g_1 + ... + g_r, gamma_r = exp(G_r) and S the state at the chunk start:
//
//   A_rs = exp(G_r - G_s) k_r.k_s (s < r),  T = (I + diag(beta) A)^-1          (UT transform)
//   W    = T diag(beta gamma) K,  Tb = T diag(beta)                              (WY factors)
//   P_rs = scale exp(G_r - G_s) q_r.k_s (s <= r),  Q' = scale diag(gamma) Q - P W
//   U    = Tb V - W S                       (the deltas written by the chunk's tokens)
//   O    = Q' S + (P Tb) V                  (= scale (diag(gamma) Q S + P U))
//   S   <- gamma_C S + K^T diag(exp(G_C - G)) U
//
// Everything that does not depend on S is computed by the parallel kernel gdn_tc_prep over all
// (chunk, value-head pair) units and packed, per (chunk, head), into one 128 x 192 bf16 operand
//     A1 = [ -W  | Tb   ]    (rows 0-63:   tokens; the state-update deltas U)
//          [ Q'  | P Tb ]    (rows 64-127: tokens; the outputs O)
// so that the sequential kernel gdn_tc_chain needs two MMAs per chunk:
//     D1 = A1 [S; V]              (M 128, K 128 + 64, N = dv slice)   -> U (rows 0-63), O (rows 64-127)
//     S  = gamma_C S + K^T (b U)  (M = dk 128, K 64, N = dv slice),  b_r = exp(G_C - G_r)
// The fp32 state lives in TMEM for the whole sequence; its bf16 copy in shared memory is the B
// operand of the next D1.  Decay ratios are always exp(G_r - G_s) with s <= r (never 1/gamma).
// Tokens past the end of a sequence inside its last chunk get beta = g = 0, which makes their rows
// of U exactly zero, so partial chunks are exact; their outputs are not stored.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int kC = 64;                      // chunk length
constexpr int kD = 128;                     // dk = dv
constexpr uint32_t kA1Bytes = 3u * 128u * 128u;  // 3 panels x 128 rows x 128 B
constexpr int kVecFloats = 128;             // per (chunk, head): b_r (64), gamma_C at [64]
constexpr int kSlices = 2;                  // dv slices of 64 columns per head in the chain kernel

// Sequences are laid out in "slots": chunk c of sequence i lives in slot floor(start_i / C) + i + c.
// This needs no prefix sum over the sequence lengths and stays below ceil(T_total / C) + nseq.
__device__ bool slot_lookup(const int32_t* cu, int nseq, int T_len, int slot, int& seq, long long& t0, int& n) {
    int lo = 0, hi = nseq - 1, best = -1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        long long a, b;
        seq_range(cu, mid, T_len, a, b);
        if (a / kC + mid <= slot) {
            best = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    if (best < 0) return false;
    long long a, b;
    seq_range(cu, best, T_len, a, b);
    const long long c = slot - (a / kC + best);
    if (c >= (b - a + kC - 1) / kC) return false;
    seq = best;
    t0 = a + c * kC;
    n = (int)min((long long)kC, b - t0);
    return true;
}

// ------------------------------------------------------------------ parallel intra-chunk kernel
// One CTA per (chunk, value-head pair): two 4-warp groups, group 0 for value head A and group 1 for
// value head B, sharing the chunk's K / Q tiles and their Gram matrices.  Two CTAs fit on one SM
// (shared memory <= 110 KB, 256 TMEM columns, <= 128 registers a thread), so sixteen warps per SM
// hide each other's latencies in the CUDA-core phases.
//
// Shared memory (byte offsets from a 1024-aligned base)
constexpr uint32_t P_KQ = 0;            // 2 panels (dk 0-63, 64-127) x [K rows 0-63 | Q rows 64-127]
constexpr uint32_t P_TOP = 32768;       // [-W_h | Tb_h] for both heads: 3 panels x 128 rows (B operand)
constexpr uint32_t P_Y = P_TOP;         // UT-solve scratch [2 heads][2 block rows][16][kYStride] fp32 (panel 0, before -W)
constexpr uint32_t P_HANDOFF = P_TOP + 16384;   // P_0 rows, bf16 [64][64] (panel 1, before -W)
constexpr uint32_t P_LC = 81920;        // L_h then T_h: 10 lower blocks of 16 x 16 fp32 per head, row stride 20
constexpr uint32_t P_LBLK = 16 * 20;    // floats per block
constexpr uint32_t P_SMALL = P_LC + 2 * 10 * P_LBLK * 4;   // G, beta, beta*gamma, a, c: [2][64] each; 1/|k|, 1/|q|: [64]
constexpr uint32_t P_BAR = P_SMALL + 5 * 2 * 64 * 4 + 2 * 64 * 4;
constexpr uint32_t P_SMEM = P_BAR + 64 + 1024;  // + alignment slack
constexpr int kPrepThreads = 256;
// TMEM columns: Gram D 0-63; T diag(beta gamma) (A operand) 0-31 after the Gram is read;
// [W_0; W_1] D 64-191; blockdiag(P_0, P_1) (A operand) 192-255; [-P W | P Tb] D 0-191.
constexpr uint32_t T_GRAM = 0, T_TD = 0, T_W = 64, T_AP = 192, T_PW = 0;
// Scratch of the UT solve: block rows 2 and 3 of T, columns 0-31 (16 rows each), stride 40 floats
// (conflict-free B-fragment loads, 16-byte aligned rows).
constexpr int kYStride = 40;
constexpr uint32_t kYHeadFloats = 2 * 16 * kYStride;
static_assert(2 * kYHeadFloats * 4 <= 16384, "the solve scratch lives in TOP panel 0");
// Output panel i = 3 h + p of [Q'_h | P_h Tb_h] (8 KB each, after their inputs are consumed)
__device__ __forceinline__ uint32_t bot_panel(int i) { return i < 4 ? P_KQ + 8192u * i : P_LC + 8192u * (i - 4); }
static_assert(P_LC + 2 * 8192 <= P_SMALL, "two output panels must fit in the L/T region");
static_assert(P_SMEM <= 113 * 1024, "two CTAs per SM");

__device__ __forceinline__ int lblk(int I, int J) { return I * (I + 1) / 2 + J; }   // J <= I

// x rounded to tf32 (10 fraction bits), to nearest with ties away from zero, by integer operations on
// its bit pattern: half a tf32 ulp (bit 12) is added to the magnitude and the 13 low bits cleared.
__device__ __forceinline__ uint32_t tf32_rna(float x) { return (__float_as_uint(x) + 0x1000u) & 0xffffe000u; }

__device__ __forceinline__ void mma_tf32_m16n8k8(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc (a 16 x 8 accumulator fragment) += A B, A 16 x 16 and B 16 x 8 fp32 in shared memory with row
// strides as and bs (B points at its first column).  Fragment g = lane / 4, t = lane % 4: A holds
// (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4) of each 8-wide k slice; B holds (k = t, n = g),
// (k = t + 4, n = g); the accumulator holds (g, 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1).
__device__ __forceinline__ void tile_mma_16x8(float (&acc)[4], const float* A, int as, const float* B, int bs,
                                              int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int kk = 0; kk < 16; kk += 8) {
        const uint32_t a[4] = {tf32_rna(A[g * as + kk + t]), tf32_rna(A[(g + 8) * as + kk + t]),
                               tf32_rna(A[g * as + kk + t + 4]), tf32_rna(A[(g + 8) * as + kk + t + 4])};
        const uint32_t b[2] = {tf32_rna(B[(kk + t) * bs + g]), tf32_rna(B[(kk + t + 4) * bs + g])};
        mma_tf32_m16n8k8(acc, a, b);
    }
}

// Store sign * acc (a 16 x 8 fragment) at D (its first column), row stride ds.
__device__ __forceinline__ void tile_store_16x8(float* D, int ds, const float (&acc)[4], float sign, int lane) {
    const int g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2*>(D + g * ds + 2 * t) = make_float2(sign * acc[0], sign * acc[1]);
    *reinterpret_cast<float2*>(D + (g + 8) * ds + 2 * t) = make_float2(sign * acc[2], sign * acc[3]);
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void named_barrier_arrive(int id, int threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// T = (I + L)^-1 of one head in place, by one 4-warp group (gw = warp in the group, bar = the group's
// named barrier).  With 16 x 16 blocks L_IJ (I, J = 0..3) and the 2 x 2 split into 32 x 32 halves:
//   (a) the diagonal blocks T_II by forward substitution in fp32 (warps 0, 1: one column a thread);
//   (b) inside each half, T_10 = -T_11 L_10 T_00 (warp 0) and T_32 = -T_33 L_32 T_22 (warp 1) -- each
//       warp uses only the blocks it has just inverted, so only warp-level syncs are needed;
//   (c) the off-diagonal half T[2:4, 0:2] = -T[2:4, 2:4] Y with Y = L[2:4, 0:2] T[0:2, 0:2], one warp
//       per (block column j, 8-column half): Y_2j, Y_3j, then T_2j = -T_22 Y_2j and
//       T_3j = -(T_32 Y_2j + T_33 Y_3j), kept in the scratch Yh (block rows 2, 3; columns 0-31).
// The off-diagonal block products run on the warp-level tensor-core MMA (m16n8k8, tf32 inputs rounded
// to nearest, fp32 accumulation): tcgen05 has no 16-row shape, and T is rounded to bf16 right after (as
// the W and T diag(beta) operands), far coarser than tf32.
__device__ __forceinline__ void unit_lower_inverse(float* L, float* Yh, int gw, int lane, int bar) {
    if (gw < 2) {
        {   // (a) column j of the diagonal block I: this warp holds blocks 2 gw and 2 gw + 1
            const int I = 2 * gw + (lane >> 4), j = lane & 15;
            float* D = L + lblk(I, I) * P_LBLK;
            float tc[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float* Dr = D + r * 20;
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int s = 0; s + 1 < r; s += 2) {
                    a0 = fmaf(Dr[s], tc[s], a0);
                    a1 = fmaf(Dr[s + 1], tc[s + 1], a1);
                }
                if (r & 1) a0 = fmaf(Dr[r - 1], tc[r - 1], a0);
                tc[r] = (r < j) ? 0.f : (r == j ? 1.f : -(a0 + a1));
            }
            __syncwarp();   // every lane of the block has read D
#pragma unroll
            for (int r = 0; r < 16; ++r) D[r * 20 + j] = tc[r];
            __syncwarp();
        }
        {   // (b) X = L_{i+1,i} T_ii into the scratch, then T_{i+1,i} = -T_{i+1,i+1} X over L_{i+1,i}
            const int i = 2 * gw;
            float* X = Yh + (uint32_t)gw * 16 * kYStride;   // block row 2 + gw of the scratch, free until (c)
            float* Lo = L + lblk(i + 1, i) * P_LBLK;
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                tile_mma_16x8(acc, Lo, 20, L + lblk(i, i) * P_LBLK + 8 * nh, 20, lane);
                tile_store_16x8(X + 8 * nh, kYStride, acc, 1.f, lane);
            }
            __syncwarp();   // X complete; every lane has finished reading L_{i+1,i}
            const float* Td = L + lblk(i + 1, i + 1) * P_LBLK;
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                tile_mma_16x8(acc, Td, 20, X + 8 * nh, kYStride, lane);
                tile_store_16x8(Lo + 8 * nh, 20, acc, -1.f, lane);
            }
        }
    }
    // T_00, T_10, T_11, T_22, T_32, T_33 are final (literal barrier ids keep the kernel at two barriers)
    if (bar == 1)
        named_barrier_sync(1, 128);
    else
        named_barrier_sync(2, 128);
    {   // (c) block column j, columns 8 nh .. 8 nh + 7 of it
        const int j = gw >> 1, nh = gw & 1;
        float* Y2 = Yh + 16 * j + 8 * nh;
        float* Y3 = Yh + 16 * kYStride + 16 * j + 8 * nh;
        const float* T1j = L + lblk(1, j) * P_LBLK + 8 * nh;   // T_10 or T_11
        float y2[4] = {0.f, 0.f, 0.f, 0.f}, y3[4] = {0.f, 0.f, 0.f, 0.f};
        if (j == 0) {   // T_01 = 0
            const float* T00 = L + lblk(0, 0) * P_LBLK + 8 * nh;
            tile_mma_16x8(y2, L + lblk(2, 0) * P_LBLK, 20, T00, 20, lane);
            tile_mma_16x8(y3, L + lblk(3, 0) * P_LBLK, 20, T00, 20, lane);
        }
        tile_mma_16x8(y2, L + lblk(2, 1) * P_LBLK, 20, T1j, 20, lane);
        tile_mma_16x8(y3, L + lblk(3, 1) * P_LBLK, 20, T1j, 20, lane);
        tile_store_16x8(Y2, kYStride, y2, 1.f, lane);
        tile_store_16x8(Y3, kYStride, y3, 1.f, lane);
        __syncwarp();   // this warp's columns of Y_2j and Y_3j are complete
        float t2[4] = {0.f, 0.f, 0.f, 0.f}, t3[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mma_16x8(t2, L + lblk(2, 2) * P_LBLK, 20, Y2, kYStride, lane);
        tile_mma_16x8(t3, L + lblk(3, 2) * P_LBLK, 20, Y2, kYStride, lane);
        tile_mma_16x8(t3, L + lblk(3, 3) * P_LBLK, 20, Y3, kYStride, lane);
        __syncwarp();   // every lane has read its Y columns
        tile_store_16x8(Y2, kYStride, t2, -1.f, lane);
        tile_store_16x8(Y3, kYStride, t3, -1.f, lane);
    }
}

__global__ void __launch_bounds__(kPrepThreads, 2)
tc_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const bf16* __restrict__ g, const bf16* __restrict__ beta, const int32_t* __restrict__ cu,
               int nseq, int T_len, int Hqk, int Hv, float scale, uint8_t* __restrict__ ws_a1,
               float* __restrict__ ws_vec, unsigned* status, const float* __restrict__ A_log,
               const float* __restrict__ dt_bias, int normalize) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float* sG = reinterpret_cast<float*>(sm + P_SMALL);   // [2][64] cumulative log decay G_r
    float* sBeta = sG + 128;                              // [2][64]
    float* sBG = sG + 256;                                // [2][64] beta_r * gamma_r
    float* sA = sG + 384;                                 // [2][64] exp(G_r - G_0)
    float* sC = sG + 512;                                 // [2][64] exp(G_0 - G_s)
    float* sRK = sG + 640;                                // [64] 1/|k_r| (1 unless normalising)
    float* sRQ = sG + 704;                                // [64] 1/|q_r|
    float* sLC = reinterpret_cast<float*>(sm + P_LC);
    const uint32_t bar_tma = sb + P_BAR, bar_mma = sb + P_BAR + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + P_BAR + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + P_BAR + 20);
    int* sFactor = reinterpret_cast<int*>(sm + P_BAR + 24);   // [2]: decay ratios factorise safely
    const uint32_t bar_drain = sb + P_BAR + 32;
    // Once every CTA of this grid has started, the chain grid that follows may take the SMs that free
    // up and run its set-up; it waits for this grid's completion before it reads the workspace.
    griddep_launch_dependents();

    const int slot = blockIdx.x, pair = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hg = warp >> 2;                            // the group's value head: 0 = hA, 1 = hB
    const int R = tid & 127;                             // TMEM lane = accumulator row of this thread
    int seq;
    long long t0;
    int n;
    if (!slot_lookup(cu, nseq, T_len, slot, seq, t0, n)) return;  // unused slot (uniform per CTA)
    // value-head pair of this CTA: the heads of one query/key head, two at a time; with an odd number
    // per query/key head the last one pairs with itself (both halves compute it and store the same bytes)
    const int G = Hv / Hqk, ppq = (G + 1) / 2;
    const int hk = pair / ppq, jp = pair % ppq;
    const int hA = hk * G + 2 * jp, hB = min(hA + 1, hk * G + G - 1);
    const int hOwn = hg == 0 ? hA : hB;
    if (tid == 0) {   // barriers first, then the K / Q tile loads, so their latency overlaps the set-up
        *abort_flag = 0;
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
        mbar_arrive_expect_tx(bar_tma, 4 * 8192);
        for (int p = 0; p < 2; ++p) {
            tma_load_3d(sb + P_KQ + p * 16384, &tm_k, 64 * p, hk, (int)t0, bar_tma);
            tma_load_3d(sb + P_KQ + p * 16384 + 8192, &tm_q, 64 * p, hk, (int)t0, bar_tma);
        }
    }
    // gates of value head hA (warp 0) / hB (warp 1), two tokens per lane; padded tokens get g = beta = 0
    float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
    if (warp < 2) {
        const int r0 = 2 * lane, r1 = 2 * lane + 1;
        const int hw = warp == 0 ? hA : hB;
        if (r0 < n) {
            g0 = __bfloat162float(g[(size_t)(t0 + r0) * Hv + hw]);
            b0 = __bfloat162float(beta[(size_t)(t0 + r0) * Hv + hw]);
        }
        if (r1 < n) {
            g1 = __bfloat162float(g[(size_t)(t0 + r1) * Hv + hw]);
            b1 = __bfloat162float(beta[(size_t)(t0 + r1) * Hv + hw]);
        }
        if (A_log) {   // raw projections a, b: form the gates (padded tokens keep g = beta = 0)
            const float al = A_log[hw], db = dt_bias[hw];
            if (r0 < n) gates_from_raw(g0, b0, al, db, g0, b0);
            if (r1 < n) gates_from_raw(g1, b1, al, db, g1, b1);
        }
    }

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tc_fence_before();
    }
    __syncthreads();   // also publishes the barrier initialisation to every thread
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);   // this warp's TMEM lane quarter

    if (warp < 2) {   // G = inclusive scan of g over the chunk
        const int hh = warp;
        const int r0 = 2 * lane, r1 = 2 * lane + 1;
        float p = g0 + g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, p, o);
            if (lane >= o) p += y;
        }
        sG[hh * 64 + r1] = p;
        sG[hh * 64 + r0] = p - g1;
        sBeta[hh * 64 + r0] = b0;
        sBeta[hh * 64 + r1] = b1;
        const float G0 = __shfl_sync(0xffffffffu, p - g1, 0), Gl = __shfl_sync(0xffffffffu, p, 31);
        if (lane == 0) sFactor[hh] = (G0 - Gl) < 80.f;
    }
    __syncthreads();
    if (tid < 128) {
        const int hh = tid >> 6, r = tid & 63;
        const float Gr = sG[hh * 64 + r], Gl = sG[hh * 64 + 63], G0 = sG[hh * 64];
        sBG[hh * 64 + r] = sBeta[hh * 64 + r] * __expf(Gr);
        sA[hh * 64 + r] = __expf(Gr - G0);
        sC[hh * 64 + r] = __expf(G0 - Gr);
        float* vec = ws_vec + ((size_t)slot * Hv + (hh == 0 ? hA : hB)) * kVecFloats;
        if (!normalize) vec[r] = __expf(Gl - Gr);   // with normalisation: written once 1/|k_r| is known
        if (r == 0) vec[64] = __expf(Gl);
    }

    // ---- [K; Q] K^T : rows 0-63 K K^T, rows 64-127 Q K^T
    mbar_wait_bounded(bar_tma, 0, abort_flag, status, kStatusTimeout, kWaitLimitNs);
    // shared-memory descriptors built once; (address >> 4) < 2^14 in this CTA, so a byte offset o moves
    // a descriptor by o >> 4 without a carry
    const uint64_t dKQk = smem_desc(sb + P_KQ, 16, 1024), dKQm = smem_desc(sb + P_KQ, 16384, 1024),
                   dTOP = smem_desc(sb + P_TOP, 16384, 1024);
    if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint64_t d = dKQk + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4);
            mma_bf16(tmem + T_GRAM, d, d, idesc_bf16(128, 64, 0, 0), ks > 0);
        }
        mma_commit(bar_mma);
    }
    __syncthreads();   // gate scalars visible to all
    mbar_wait_bounded(bar_mma, 0, abort_flag, status, kStatusTimeout, kWaitLimitNs);
    tc_fence_after();
    {
        // row R of the Gram; group hg builds the rows of its own head
        uint32_t a[64];
        tmem_ld32(tl + T_GRAM, *reinterpret_cast<uint32_t(*)[32]>(a));
        tmem_ld32(tl + T_GRAM + 32, *reinterpret_cast<uint32_t(*)[32]>(a + 32));
        tmem_wait_ld();
        if (normalize) {   // l2 normalisation of q and k folded into per-row scalars (eps 1e-6)
            if (R < 64) {
                float kk = 0.f;   // k_r . k_r is the diagonal of K K^T
#pragma unroll
                for (int s = 0; s < 64; ++s) kk = (s == R) ? __uint_as_float(a[s]) : kk;
                const float rk = rsqrtf(kk + 1e-6f);
                if (hg == 0) sRK[R] = rk;
                ws_vec[((size_t)slot * Hv + hOwn) * kVecFloats + R] = __expf(sG[hg * 64 + 63] - sG[hg * 64 + R]) * rk;
                sBG[hg * 64 + R] *= rk;
            } else if (hg == 0) {
                const int r = R - 64;
                float qq = 0.f;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint4 qv = *reinterpret_cast<const uint4*>(sm + P_KQ + (c >> 3) * 16384 + 8192 + swz(r, c & 7));
                    const bf16* qe = reinterpret_cast<const bf16*>(&qv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) qq = fmaf(__bfloat162float(qe[e]), __bfloat162float(qe[e]), qq);
                }
                sRQ[r] = rsqrtf(qq + 1e-6f);
            }
        } else if (tid < 64) {
            sRK[tid] = 1.f;
            sRQ[tid] = 1.f;
        }
        __syncthreads();
        if (normalize) {   // fold 1/|k_s| into the column factor exp(G_0 - G_s) once
            if (tid < 128) sC[tid] *= sRK[tid & 63];
            __syncthreads();
        }
        const float* Gh = sG + hg * 64;
        const float* ch = sC + hg * 64;
        const bool fac = sFactor[hg] != 0;
        if (R < 64) {   // row r of K K^T -> L_h[r][s] = beta_r exp(G_r - G_s) k_r.k_s (s < r), lower blocks
            const int r = R, I = r >> 4, rr = r & 15;
            const float br = sBeta[hg * 64 + r] * sRK[r], ar = sA[hg * 64 + r], Gr = Gh[r];
            float* Lh = sLC + hg * 10 * P_LBLK;
            const float rowc = br * ar;   // factorised decay: beta_r exp(G_r - G_0) / |k_r|
            for (int J = 0; J <= I; ++J) {
                float* dst = Lh + lblk(I, J) * P_LBLK + rr * 20;
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    float o[4];
                    if (fac) {   // uniform per head: exp(G_0 - G_s) / |k_s| is the column factor ch[s]
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s = 16 * J + 4 * s4 + e;
                            o[e] = (s < r) ? rowc * __uint_as_float(a[s]) * ch[s] : 0.f;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s = 16 * J + 4 * s4 + e;
                            o[e] = (s < r) ? br * __expf(Gr - Gh[s]) * __uint_as_float(a[s]) * sRK[s] : 0.f;
                        }
                    }
                    *reinterpret_cast<float4*>(dst + 4 * s4) = make_float4(o[0], o[1], o[2], o[3]);
                }
            }
        } else {        // row r of Q K^T -> P_h[r][s] = scale exp(G_r - G_s) q_r.k_s (s <= r)
            const int r = R - 64;
            const float sq = scale * sRQ[r];
            const float ar = sA[hg * 64 + r], Gr = Gh[r];
            uint32_t w[32];
            if (fac) {   // uniform per head
                const float rowc = sq * ar;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float pv[2];
#pragma unroll
                    for (int f = 0; f < 2; ++f) {
                        const int s = 2 * e + f;
                        pv[f] = (s <= r) ? rowc * __uint_as_float(a[s]) * ch[s] : 0.f;
                    }
                    w[e] = pack_bf16(pv[0], pv[1]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float pv[2];
#pragma unroll
                    for (int f = 0; f < 2; ++f) {
                        const int s = 2 * e + f;
                        pv[f] = (s <= r) ? sq * __expf(Gr - Gh[s]) * __uint_as_float(a[s]) * sRK[s] : 0.f;
                    }
                    w[e] = pack_bf16(pv[0], pv[1]);
                }
            }
            if (hg == 1) {   // own lane: [0 | P_1 row] (the zero half is written by group 0)
                tmem_st32(tl + T_AP + 32, w);
            } else {         // P_0 row r belongs to lane r: hand it over through shared memory, 16-byte
                             // chunk c of row r at chunk c ^ (r % 8) (eight consecutive rows: all banks)
                uint4* dst = reinterpret_cast<uint4*>(sm + P_HANDOFF + r * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c ^ (r & 7)] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
#pragma unroll
                for (int e = 0; e < 32; ++e) w[e] = 0u;
                tmem_st32(tl + T_AP, w);
            }
        }
    }
    __syncthreads();
    if (R < 64) {   // lanes 0-63: [P_0 row | 0], the halves written by the two groups
        uint32_t w[32];
        if (hg == 0) {
            const uint4* src = reinterpret_cast<const uint4*>(sm + P_HANDOFF + R * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 x = src[c ^ (R & 7)];
                w[4 * c] = x.x; w[4 * c + 1] = x.y; w[4 * c + 2] = x.z; w[4 * c + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) w[e] = 0u;
        }
        tmem_st32(tl + T_AP + 32 * hg, w);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();

    // ---- T_h = (I + L_h)^-1 in place (group hg, head hg); then T_h diag(beta gamma) -> TMEM (A
    // operand) and T_h diag(beta) -> TOP panel 2, the two groups taking 32 columns each
    unit_lower_inverse(sLC + hg * 10 * P_LBLK, reinterpret_cast<float*>(sm + P_Y) + hg * kYHeadFloats, warp & 3,
                       lane, 1 + hg);
    __syncthreads();
    {
        const int hh = R >> 6, r = R & 63, I = r >> 4, rr = r & 15;
        const float* Th = sLC + hh * 10 * P_LBLK;
        const float* Yh = reinterpret_cast<const float*>(sm + P_Y) + hh * kYHeadFloats;
        const float* dg = sBG + hh * 64;
        const float* bt = sBeta + hh * 64;
        uint32_t wd[16];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int J = 2 * hg + jj;
#pragma unroll
            for (int c = 0; c < 2; ++c) {   // 8 columns s = 16 J + 8 c ..
                float tv[8];
                if (J <= I) {
                    // blocks (2|3, 0|1) of T are in the scratch, the others in place of L
                    const float* src = (I >= 2 && J <= 1) ? Yh + ((I - 2) * 16 + rr) * kYStride + 16 * J + 8 * c
                                                          : Th + lblk(I, J) * P_LBLK + rr * 20 + 8 * c;
                    const float4 x0 = *reinterpret_cast<const float4*>(src), x1 = *reinterpret_cast<const float4*>(src + 4);
                    tv[0] = x0.x; tv[1] = x0.y; tv[2] = x0.z; tv[3] = x0.w;
                    tv[4] = x1.x; tv[5] = x1.y; tv[6] = x1.z; tv[7] = x1.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) tv[e] = 0.f;
                }
                const int s0 = 16 * J + 8 * c;
                // eight consecutive column factors in two 16-byte loads (the vectors are 256-byte aligned)
                float dgv[8], btv[8];
                *reinterpret_cast<float4*>(dgv) = *reinterpret_cast<const float4*>(dg + s0);
                *reinterpret_cast<float4*>(dgv + 4) = *reinterpret_cast<const float4*>(dg + s0 + 4);
                *reinterpret_cast<float4*>(btv) = *reinterpret_cast<const float4*>(bt + s0);
                *reinterpret_cast<float4*>(btv + 4) = *reinterpret_cast<const float4*>(bt + s0 + 4);
                uint32_t wb[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    wd[8 * jj + 4 * c + e] = pack_bf16(tv[2 * e] * dgv[2 * e], tv[2 * e + 1] * dgv[2 * e + 1]);
                    wb[e] = pack_bf16(tv[2 * e] * btv[2 * e], tv[2 * e + 1] * btv[2 * e + 1]);
                }
                *reinterpret_cast<uint4*>(sm + P_TOP + 2 * 16384 + swz(R, s0 >> 3)) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
            }
        }
        tmem_st16(tl + T_TD + 16 * hg, wd);
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- [W_0; W_1] = [T_0 D_0; T_1 D_1] K
    if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_ta(tmem + T_W, tmem + T_TD + 8 * ks, dKQm + ((ks * 2048) >> 4), idesc_bf16(128, 128, 0, 1), ks > 0);
        mma_commit(bar_mma);
    }
    mbar_wait_bounded(bar_mma, 1, abort_flag, status, kStatusTimeout, kWaitLimitNs);
    tc_fence_after();
    {   // row R of [W_0; W_1] -> -W in TOP panel hg (columns 64 hg .. 64 hg + 63)
        uint8_t* pan = sm + P_TOP + hg * 16384;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
            uint32_t a[32];
            tmem_ld32(tl + T_W + 64 * hg + 32 * cc, a);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16(-__uint_as_float(a[8 * c + 2 * e]), -__uint_as_float(a[8 * c + 2 * e + 1]));
                *reinterpret_cast<uint4*>(pan + swz(R, cc * 4 + c)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- blockdiag(P_0, P_1) [-W | Tb]: -P W and P Tb for both heads
    if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ta(tmem + T_PW, tmem + T_AP + 8 * ks, dTOP + ((ks * 2048) >> 4), idesc_bf16(128, 192, 0, 1), ks > 0);
        mma_commit(bar_mma);
        // the [-W | Tb] rows of A1 are final (they are this MMA's B operand): their stores read the same
        // shared memory while the MMA runs, and issuing them here keeps the issue off the barrier below
        for (int h = 0; h < 2; ++h) {
            uint8_t* dst = ws_a1 + ((size_t)slot * Hv + (h == 0 ? hA : hB)) * kA1Bytes;
            for (int p = 0; p < 3; ++p) bulk_s2g(dst + p * 16384, sb + P_TOP + p * 16384 + h * 8192, 8192);
        }
        bulk_commit();
    }
    // this thread's query row, the 64 features its group needs (columns 32 cb .. of the panels 0, 1 of
    // the output rows, cb = hg, hg + 2), read before the K/Q panels are reused for the outputs
    const int hh = R >> 6, r = R & 63;
    uint4 qrow[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        qrow[c] = *reinterpret_cast<const uint4*>(sm + P_KQ + (c >> 2) * 16384 + 8192 + swz(r, 4 * hg + (c & 3)));
    mbar_wait_bounded(bar_mma, 0, abort_flag, status, kStatusTimeout, kWaitLimitNs);
    tc_fence_after();
    __syncthreads();   // every thread holds its q features: the K/Q panels are free
    {
        const float qs = scale * __expf(sG[hh * 64 + r]) * sRQ[r];   // scale * gamma_r / |q_r|
        // panel by panel, so that the bulk stores of the first panels drain while the later ones are built;
        // column block cb = 2 p + hg of the 192 columns is this group's half of panel p
        for (int p = 0; p < 3; ++p) {
            const int cb = 2 * p + hg;
            uint32_t a[32];
            tmem_ld32(tl + T_PW + 32 * cb, a);
            tmem_wait_ld();
            uint8_t* pan = sm + bot_panel(3 * hh + p);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t chunk = hg * 4 + c;
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(a[8 * c + e]);
                if (p < 2) {   // Q' = scale gamma_r q_r - P W
                    const bf16* qe = reinterpret_cast<const bf16*>(&qrow[p * 4 + c]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = fmaf(qs, __bfloat162float(qe[e]), x[e]);
                }
                *reinterpret_cast<uint4*>(pan + swz(r, chunk)) =
                    make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
            }
            fence_proxy_async_smem();
            if (p == 2) tc_fence_before();   // every TMEM read of this CTA precedes the deallocation
            __syncthreads();
            if (tid == 0) {   // panel p of A1 for each head: [TOP rows of the head | output rows of the head]
                for (int h = 0; h < 2; ++h)
                    bulk_s2g(ws_a1 + ((size_t)slot * Hv + (h == 0 ? hA : hB)) * kA1Bytes + p * 16384 + 8192,
                             sb + bot_panel(3 * h + p), 8192);
                bulk_commit();
            }
        }
    }
    if (warp == 0) {
        if (tid == 0) {
            bulk_wait_read();   // shared memory may be released; the global writes finish on their own
            if (*abort_flag) {   // a bounded wait gave up: no MMA or tile load of this CTA may still be running
                mbar_init(bar_drain, 1);   // initialised only here: off the normal path
                mbar_fence_init();
                mma_commit(bar_drain);
                mbar_wait_drain(bar_drain, 0, kWaitLimitNs);
                mbar_wait_drain(bar_tma, 0, kWaitLimitNs);
            }
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------------ sequential chain kernel
constexpr uint32_t C_A1 = 0;            // 2 stages x 48 KB
constexpr uint32_t C_VT = 98304;        // 2 stages x 8 KB  (V slice: 1 panel x 64 token rows)
constexpr uint32_t C_KT = 114688;       // 3 stages x 16 KB (K tile: 2 panels x 64 token rows)
constexpr uint32_t C_SB = 163840;       // bf16 state slice: 1 panel x 128 dk rows
constexpr uint32_t C_UB = 180224;       // bf16 b*U: 1 panel x 64 token rows
constexpr uint32_t C_VEC = 188416;      // 3 stages x 512 B
constexpr uint32_t C_OST = 190464;      // output rows of a full chunk, 3 buffers x 64 token rows x 64 bf16 (swizzled)
constexpr uint32_t C_BAR = C_OST + 3 * 8192;
constexpr uint32_t C_SMEM = C_BAR + 128 + 1024;
constexpr int kKStages = 3;
// Operands arrive in two rings freed at different times: A1 and the V slice (2 stages, consumed by
// D1) and the K tile with the b / gamma_C vector (3 stages, consumed by the state update and the
// epilogues).
constexpr uint32_t kStageBytesA = kA1Bytes + 8192;
constexpr uint32_t kStageBytesK = 16384 + kVecFloats * 4;
// 9 warps.  Warps 0-7 are the epilogue warps: warps w and w + 4 read TMEM lane quarter w % 4 and split
// the slice's 64 columns.  Lane 0 of warp 8 issues every MMA and does no epilogue work: an issuing
// thread that also ran an epilogue made its warp the last to reach each barrier.  Lane 0 of warp 6 (an
// output warp, with slack) issues the operand loads once the state-update barrier has passed: the
// shared-memory proxy fences of the epilogues measured several times slower while a bulk copy was
// landing in shared memory, so the copies land between the two epilogues.
constexpr int kEpilogueThreads = 256;
constexpr int kChainThreads = kEpilogueThreads + 32;
constexpr int kIssuer = kEpilogueThreads;
constexpr int kProducer = 192;
// TMEM columns: state S 0-63; D1 of even chunks 64-127, of odd chunks 128-191.


__global__ void __launch_bounds__(kChainThreads, 1)
tc_chain_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_out, const uint8_t* __restrict__ ws_a1, const float* __restrict__ ws_vec, const float* __restrict__ S0,
                bf16* __restrict__ out, float* __restrict__ S_final, const int32_t* __restrict__ cu, int nseq,
                int T_len, int Hqk, int Hv, int num_slots, unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    // bar_a[2] (A1 + V), bar_k[3] (K + vector), mma1, mma2
    const uint32_t bar_a0 = sb + C_BAR, bar_k0 = sb + C_BAR + 16, bar_mma1 = sb + C_BAR + 40,
                   bar_mma2 = sb + C_BAR + 48, bar_drain = sb + C_BAR + 64;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C_BAR + 56);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C_BAR + 60);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp < kEpilogueThreads / 32;   // an epilogue warp (warp 8 issues)
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int R = 32 * quarter + lane;      // TMEM lane = accumulator row
    const int cb = 32 * half;               // this thread's 32 of the slice's 64 columns
    const int z = blockIdx.x % kSlices;
    const int h = (blockIdx.x / kSlices) % Hv;
    const int i = blockIdx.x / (kSlices * Hv);
    const int hk = h / (Hv / Hqk);
    long long s0, s1;
    seq_range(cu, i, T_len, s0, s1);
    const long long base = s0 / kC + i;
    long long nch = (s1 - s0 + kC - 1) / kC;
    if (base + nch > num_slots) nch = max(0LL, num_slots - base);   // only for malformed offsets

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tc_fence_before();
    }
    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar_a0, 1);
        mbar_init(bar_a0 + 8, 1);
        for (int q = 0; q < kKStages; ++q) mbar_init(bar_k0 + 8 * q, 1);
        mbar_init(bar_mma1, 1);
        mbar_init(bar_mma2, 1);
        mbar_fence_init();
    }
    const size_t srow = (((size_t)i * Hv + h) * kD + R) * kD + 64 * z + cb;   // 32 floats of state row R
    // S0 is an input: its rows are read while the prep grid may still be running.  Everything that
    // reads the prep's workspace (or writes memory) comes after griddep_wait below.
    uint32_t s0v[32];
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
        const float4 x = (S0 && epi) ? *reinterpret_cast<const float4*>(S0 + srow + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        s0v[e] = __float_as_uint(x.x); s0v[e + 1] = __float_as_uint(x.y);
        s0v[e + 2] = __float_as_uint(x.z); s0v[e + 3] = __float_as_uint(x.w);
    }
    __syncthreads();
    tc_fence_after();
    griddep_wait();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);

    auto wait_a = [&](long long c) {
        return mbar_wait_bounded(bar_a0 + 8 * (uint32_t)(c & 1), (uint32_t)((c >> 1) & 1), abort_flag, status,
                                 kStatusTimeout, kWaitLimitNs);
    };
    auto wait_k = [&](long long c) {
        return mbar_wait_bounded(bar_k0 + 8 * (uint32_t)(c % kKStages), (uint32_t)((c / kKStages) & 1), abort_flag,
                                 status, kStatusTimeout, kWaitLimitNs);
    };
    // A stage is refilled only by a thread whose own waits showed it consumed (a register test: a
    // shared-memory read of the abort flag here added ~8 us to the 8k prefill's chain), so after a bounded
    // wait gives up no load overlaps another on a stage and the drain before exit covers every one.
    bool waits_ok = true;
    auto issue_loads_a = [&](long long c) {   // A1 and the V slice of chunk c
        if (!waits_ok) return;
        const int st = (int)(c & 1);
        const long long slot = base + c;
        const uint32_t bar = bar_a0 + 8 * st;
        mbar_arrive_expect_tx(bar, kStageBytesA);
        bulk_g2s(sb + C_A1 + st * kA1Bytes, ws_a1 + ((size_t)slot * Hv + h) * kA1Bytes, kA1Bytes, bar);
        tma_load_3d(sb + C_VT + st * 8192, &tm_v, 64 * z, h, (int)(s0 + c * kC), bar);
    };
    auto issue_loads_k = [&](long long c) {   // K tile and the b / gamma_C vector of chunk c
        if (!waits_ok) return;
        const int st = (int)(c % kKStages);
        const long long slot = base + c;
        const int tc0 = (int)(s0 + c * kC);
        const uint32_t bar = bar_k0 + 8 * st;
        mbar_arrive_expect_tx(bar, kStageBytesK);
        tma_load_3d(sb + C_KT + st * 16384, &tm_k, 0, hk, tc0, bar);
        tma_load_3d(sb + C_KT + st * 16384 + 8192, &tm_k, 64, hk, tc0, bar);
        bulk_g2s(sb + C_VEC + st * 512, ws_vec + ((size_t)slot * Hv + h) * kVecFloats, kVecFloats * 4, bar);
    };
    // D1(c) = [Tb; P Tb] V_c: the part of A1 [S; V] that does not depend on the state, issued one chunk
    // ahead so it runs while the previous chunk's state update is on the critical path.
    // Shared-memory descriptors built once: the 14-bit address field holds (address >> 4) < 2^14 for
    // every operand of this CTA, so a byte offset o moves a descriptor by o >> 4 without a carry.
    const uint64_t dA1 = smem_desc(sb + C_A1, 16, 1024), dVT = smem_desc(sb + C_VT, 1024, 1024),
                   dSB = smem_desc(sb + C_SB, 1024, 1024), dKT = smem_desc(sb + C_KT, 8192, 1024),
                   dUB = smem_desc(sb + C_UB, 1024, 1024);
    auto issue_v_part = [&](long long c) {
        const int st = (int)(c & 1);
        const uint64_t a1 = dA1 + ((st * kA1Bytes + 2 * 16384) >> 4), vt = dVT + ((st * 8192) >> 4);
        const uint32_t d1 = tmem + 64 + 64 * (uint32_t)st;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16(d1, a1 + ((ks * 32) >> 4), vt + ((ks * 2048) >> 4), idesc_bf16(128, 64, 0, 1), ks > 0);
    };

    // Output rows R - 64 of chunk cc (warps of lane quarters 2-3) from its D1 buffer: a full chunk
    // goes through swizzled staging and one TMA store by warp 7; the last chunk of a sequence stores
    // its own rows (the next sequence's rows follow them).
    auto write_out = [&](long long cc) {
        const long long tcc = s0 + cc * kC;
        const int nn = (int)min((long long)kC, s1 - tcc), r = R - 64;
        uint32_t a[32];
        tmem_ld32(tl + 64 + 64 * (uint32_t)(cc & 1) + cb, a);
        tmem_wait_ld();
        tc_fence_before();
        if (nn == kC) {
            uint8_t* ost = sm + C_OST + (uint32_t)(cc % 3) * 8192;
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                const uint32_t* src = a + 8 * c8;
                *reinterpret_cast<uint4*>(ost + swz((uint32_t)r, (uint32_t)((cb >> 3) + c8))) =
                    make_uint4(pack_bf16(__uint_as_float(src[0]), __uint_as_float(src[1])),
                               pack_bf16(__uint_as_float(src[2]), __uint_as_float(src[3])),
                               pack_bf16(__uint_as_float(src[4]), __uint_as_float(src[5])),
                               pack_bf16(__uint_as_float(src[6]), __uint_as_float(src[7])));
            }
            fence_proxy_async_smem();
            named_barrier_sync(3, 128);   // the four output warps' rows are staged
            if (warp == 7 && lane == 0) {
                tma_store_3d(&tm_out, 64 * z, h, (int)tcc, sb + C_OST + (uint32_t)(cc % 3) * 8192);
                bulk_commit();
                bulk_wait_read_1();   // the store of two chunks back has read its buffer
            }
        } else if (r < nn) {
            uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)(tcc + r) * Hv + h) * kD + 64 * z + cb);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                const uint32_t* src = a + 8 * c8;
                dst[c8] = make_uint4(pack_bf16(__uint_as_float(src[0]), __uint_as_float(src[1])),
                                     pack_bf16(__uint_as_float(src[2]), __uint_as_float(src[3])),
                                     pack_bf16(__uint_as_float(src[4]), __uint_as_float(src[5])),
                                     pack_bf16(__uint_as_float(src[6]), __uint_as_float(src[7])));
            }
        }
    };

    if (nch == 0) {   // empty sequence: the final state is the initial state
        if (S_final && epi) {
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(S_final + srow + e) =
                    make_float4(__uint_as_float(s0v[e]), __uint_as_float(s0v[e + 1]), __uint_as_float(s0v[e + 2]),
                                __uint_as_float(s0v[e + 3]));
        }
    } else {
        if (tid == kIssuer) {
            for (long long c = 0; c < 2 && c < nch; ++c) issue_loads_a(c);
            for (long long c = 0; c < kKStages && c < nch; ++c) issue_loads_k(c);
        }
        // prologue: bf16 copy of S0 into SB, gamma_C(0) * S0 into TMEM, V part of chunk 0
        if (epi) {
            wait_k(0);
            const float g0 = reinterpret_cast<const float*>(sm + C_VEC)[64];   // vector of chunk 0 (K stage 0)
            uint32_t (&v)[32] = s0v;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float* f = reinterpret_cast<const float*>(v + 8 * c);
                *reinterpret_cast<uint4*>(sm + C_SB + swz(R, (cb >> 3) + c)) =
                    make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(g0 * __uint_as_float(v[e]));
            tmem_st32(tl + cb, v);
            tmem_wait_st();
        } else if (lane == 0 && wait_a(0)) {
            tc_fence_after();
            issue_v_part(0);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        uint32_t spend[32];   // gamma-scaled state row of the previous step, stored to TMEM after the next D1 issue
        for (long long c = 0; c < nch; ++c) {
            const int st = (int)(c & 1);
            const uint32_t par = (uint32_t)(c & 1);
            const long long tc0 = s0 + c * kC;
            const int n = (int)min((long long)kC, s1 - tc0);
            const uint32_t d1 = tmem + 64 + 64 * (uint32_t)st;
            const int kst = (int)(c % kKStages);
            const bool last = (c + 1 == nch);
            if (!epi) {   // ---- the issuing warp
                if (lane == 0) {   // D1 += A1[:, S part] S   (the V part is already in D1)
                    wait_a(c);
                    tc_fence_after();
                    const uint64_t a1 = dA1 + ((st * kA1Bytes) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16(d1, a1 + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4), dSB + ((ks * 2048) >> 4),
                                 idesc_bf16(128, 64, 0, 1), 1);
                    mma_commit(bar_mma1);
                }
                __syncwarp();
                named_barrier_sync(1, kChainThreads);   // b U is in shared memory, every state row in TMEM
                if (lane == 0) {   // S (gamma_C-scaled, in TMEM) += K^T (b U); then the next chunk's V part
                    tc_fence_after();
                    const uint64_t kt = dKT + ((kst * 16384) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(tmem, kt + ((ks * 2048) >> 4), dUB + ((ks * 2048) >> 4), idesc_bf16(128, 64, 1, 1), 1);
                    mma_commit(bar_mma2);
                    if (!last && wait_a(c + 1)) issue_v_part(c + 1);
                }
                __syncwarp();
            } else {      // ---- the epilogue warps
                if (c > 0) {   // TMEM columns 0-63 (the state) are not touched by the D1 MMA
                    tmem_st32(tl + cb, spend);
                    tmem_wait_st();
                    tc_fence_before();
                }
                // the previous chunk's output rows, while this chunk's D1 runs: its D1 buffer is next
                // overwritten by the V part issued after this step's state-update barrier
                if (quarter >= 2 && c > 0) write_out(c - 1);
                waits_ok &= wait_k(c);
                waits_ok &= mbar_wait_bounded(bar_mma1, par, abort_flag, status, kStatusTimeout, kWaitLimitNs);
                tc_fence_after();
                if (quarter < 2) {   // U row R scaled by b_r = exp(G_C - G_r) -> B operand of the state update
                    uint32_t a[32];
                    tmem_ld32(tl + 64 + 64 * st + cb, a);
                    tmem_wait_ld();
                    const float br = reinterpret_cast<const float*>(sm + C_VEC + kst * 512)[R];
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = br * __uint_as_float(a[8 * c8 + e]);
                        *reinterpret_cast<uint4*>(sm + C_UB + swz(R, (cb >> 3) + c8)) =
                            make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    named_barrier_arrive(1, kChainThreads);
                } else {             // the output warps (their rows are written a step later)
                    if (warp == kProducer / 32) {   // waits for the barrier, then issues the loads
                        named_barrier_sync(1, kChainThreads);
                        if (lane == 0) {
                            if (c + 2 < nch) issue_loads_a(c + 2);   // A1 and V of this stage: D1 is complete
                            // the K stage of chunk c - 1: its state update completed before the last step ended
                            if (c >= 1 && c + 2 < nch) issue_loads_k(c + 2);
                        }
                    } else {
                        named_barrier_arrive(1, kChainThreads);   // its gamma-scaled state rows are in TMEM
                    }
                }
                float gnext = 1.f;
                if (!last) {   // the next chunk's gamma_C, read while the state update runs
                    waits_ok &= wait_k(c + 1);
                    gnext = reinterpret_cast<const float*>(sm + C_VEC + (int)((c + 1) % kKStages) * 512)[64];
                }
                waits_ok &= mbar_wait_bounded(bar_mma2, par, abort_flag, status, kStatusTimeout, kWaitLimitNs);
                tc_fence_after();
                {   // new state row R: bf16 copy for the next D1 now, gamma-scaled copy to TMEM next step
                    uint32_t v[32];
                    tmem_ld32(tl + cb, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const float* f = reinterpret_cast<const float*>(v + 8 * c4);
                        *reinterpret_cast<uint4*>(sm + C_SB + swz(R, (cb >> 3) + c4)) =
                            make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
                    }
                    if (last) {
                        if (S_final) {
#pragma unroll
                            for (int e = 0; e < 32; e += 4)
                                *reinterpret_cast<float4*>(S_final + srow + e) =
                                    make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                                __uint_as_float(v[e + 3]));
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) spend[e] = __float_as_uint(gnext * __uint_as_float(v[e]));
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
            }
            __syncthreads();
        }
        if (epi && quarter >= 2) write_out(nch - 1);   // the last chunk's output rows
        if (warp == 7 && lane == 0) bulk_wait_all();   // the output stores are complete
        if (tid == kIssuer && *abort_flag) {
            // A bounded wait gave up: before the TMEM and shared memory are released, every MMA has
            // completed and no copy is still landing (consumers may have skipped chunks whose loads were
            // issued).  Each stage's last armed phase is the latest one, so its parity test is exact.
            mbar_init(bar_drain, 1);   // initialised only here: off the normal path
            mbar_fence_init();
            mma_commit(bar_drain);
            mbar_wait_drain(bar_drain, 0, kWaitLimitNs);
            for (long long c = max(0LL, nch - 2); c < nch; ++c)
                mbar_wait_drain(bar_a0 + 8 * (uint32_t)(c & 1), (uint32_t)((c >> 1) & 1), kWaitLimitNs);
            for (long long c = max(0LL, nch - kKStages); c < nch; ++c)
                mbar_wait_drain(bar_k0 + 8 * (uint32_t)(c % kKStages), (uint32_t)((c / kKStages) & 1), kWaitLimitNs);
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// [tokens, heads, 128] bf16 tensor, box of 64 tokens x 1 head x 64 features, 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, long long tokens, int heads) {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t elem[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

long long total_tokens(int B, int T, bool packed) { return packed ? (long long)T : (long long)B * T; }
long long num_slots(long long ttot, int nseq) { return (ttot + kC - 1) / kC + nseq; }

void record_event(void** events, int num_events, int idx, cudaStream_t s) {
    if (events && idx < num_events && events[idx]) cudaEventRecord(static_cast<cudaEvent_t>(events[idx]), s);
}

}  // namespace

// The chunk length the caller asks for (16, 32 or 64) is a blocking choice: every chunk length gives the
// token loop's result up to rounding, and the tensor-core tiles of this path hold 64-token chunks, so
// it serves all three with C = 64.
bool tc_prefill_eligible(int dtype, int dk, int dv, int Hqk, int Hv, int chunk, unsigned flags) {
    (void)flags;   // normalisation and raw gates are handled inside the kernels
    (void)chunk;
    return dtype == GDN_BF16 && dk == kD && dv == kD;
}

size_t tc_prefill_workspace_bytes(int B, int T, int Hv, int num_seqs, bool packed) {
    const long long slots = num_slots(total_tokens(B, T, packed), num_seqs);
    const size_t a1 = (size_t)slots * Hv * kA1Bytes;
    const size_t vec = (size_t)slots * Hv * kVecFloats * sizeof(float);
    return a1 + vec;
}

void* tensor_map_encoder() {
    static std::once_flag once;
    static void* fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = f;
    });
    return fn;
}

// Kernel attributes (shared-memory size and carveout) belong to a device: set them once per device.
cudaError_t set_kernel_attributes() {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static bool done[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(tc_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_SMEM);
    if (e == cudaSuccess)   // two prep CTAs per SM need the largest shared-memory carveout
        e = cudaFuncSetAttribute(tc_prep_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C_SMEM);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

cudaError_t launch_tc_prefill(const PrefillArgs& a, void** events, int num_events) {
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    if ((e = set_kernel_attributes()) != cudaSuccess) return e;

    const bool packed = a.cu_seqlens != nullptr;
    const long long ttot = total_tokens(a.B, a.T, packed);
    const long long slots = num_slots(ttot, a.num_seqs);
    if (ttot > INT32_MAX || slots > INT32_MAX) return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv, to;
    if ((e = make_map(&tq, a.q, ttot, a.Hqk)) != cudaSuccess) return e;
    if ((e = make_map(&tk, a.k, ttot, a.Hqk)) != cudaSuccess) return e;
    if ((e = make_map(&tv, a.v, ttot, a.Hv)) != cudaSuccess) return e;
    if ((e = make_map(&to, a.out, ttot, a.Hv)) != cudaSuccess) return e;
    uint8_t* ws_a1 = static_cast<uint8_t*>(a.workspace);
    float* ws_vec = reinterpret_cast<float*>(ws_a1 + (size_t)slots * a.Hv * kA1Bytes);
    const int T_len = a.T;

    record_event(events, num_events, 0, a.stream);
    const int G = a.Hv / a.Hqk;   // value heads per query/key head, processed two at a time
    tc_prep_kernel<<<dim3((unsigned)slots, (unsigned)(a.Hqk * ((G + 1) / 2))), kPrepThreads, P_SMEM, a.stream>>>(
        tq, tk, static_cast<const bf16*>(a.g), static_cast<const bf16*>(a.beta), a.cu_seqlens, a.num_seqs, T_len,
        a.Hqk, a.Hv, a.scale, ws_a1, ws_vec, a.status, (a.flags & GDN_RAW_GATES) ? a.A_log : nullptr, a.dt_bias,
        (a.flags & GDN_NORMALIZE_QK) ? 1 : 0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // The chain follows the prep with programmatic stream serialisation: its CTAs take the SMs freed by the
    // prep's last wave and run their set-up there.  Not when an event is recorded between the two.
    const bool mid_event = events && num_events > 1 && events[1];
    record_event(events, num_events, 1, a.stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)a.num_seqs * a.Hv * kSlices));
    cfg.blockDim = dim3(kChainThreads);
    cfg.dynamicSmemBytes = C_SMEM;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = mid_event ? 0 : 1;
    e = cudaLaunchKernelEx(&cfg, tc_chain_kernel, tk, tv, to, (const uint8_t*)ws_a1, (const float*)ws_vec, a.S0,
                           static_cast<bf16*>(a.out), a.S_final, a.cu_seqlens, a.num_seqs, T_len, a.Hqk, a.Hv,
                           (int)slots, a.status);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    record_event(events, num_events, 2, a.stream);
    return cudaSuccess;
}

}  // namespace gdn
