// The backward pass's forward chunk chain on the sm_103a tensor cores (tcgen05.mma kind::f16, fp32
// accumulators in TMEM), in fp32 accuracy, for bf16 k and dk = dv = 128.
//
// Per (sequence, value head, 64-column slice of dv), chunk by chunk (C = 64 tokens; the chunk algebra
// of the backward kernels: W = T diag(beta gamma) K and U~ = T diag(beta) V from the WY kernel, S the
// state at the chunk start, b_r = exp(G_C - G_r), times 1/|k_r| with in-kernel normalisation):
//     U = U~ - W S                     (to the workspace, over U~; the chunk-local kernel reads it)
//     S <- gamma_C S + K^T diag(b) U   (the chunk-start states go to the workspace)
// which is the update of "Transformer by Hand, ch. 7", section "The formula", regrouped by chunks.
//
// fp32 accuracy from bf16 MMAs: every fp32 operand x is split into three bf16 parts x = h + m + l
// exactly (h = x cut to its leading 8 significand bits, m = (x - h) cut the same way, l = x - h - m;
// both differences are exact in fp32 and l has at most 8 significand bits; integer masks, no
// conversion instructions), and products are sums of part products in fp32 accumulators.  K is a
// bf16 input (exact), so
//     K^T diag(b) U = K^T (bU)_h + K^T (bU)_m + K^T (bU)_l                (3 MMA groups of 4)
// and for W S, the 64-row W parts are stacked to fill the 128 TMEM lanes of one M = 128 product:
//     D = [W_h; W_m] (S_h + S_m + S_l) + [W_l; 0] S_h                       (4 groups of 8)
// whose rows r and r + 64 add up to W S but for W_l (S_m + S_l), below 2^-22 |W| |S|.
//
// Data movement: K tiles, W (with the decay sums G) and U~ arrive by TMA a chunk or two ahead; U and
// the chunk-start states leave by TMA tensor stores from swizzled staging, so that no thread stores
// a row of its own to global memory (a warp of row-owning threads touched 32 cache lines per store).
// Every wait is bounded (2 s), as in the forward kernels.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int kC = 64, kD = 128, kSW = 64;   // chunk, head dim, dv slice of one CTA
constexpr int kSlices = kD / kSW;
// Shared memory (byte offsets from a 1024-aligned base)
constexpr uint32_t B_SB = 0;          // S parts h, m, l: MN-major B, 128 dk rows x 64 columns (16 KB each)
constexpr uint32_t B_UB = 49152;      // (bU) parts h, m, l: MN-major B, 64 token rows x 64 columns (8 KB each)
constexpr uint32_t B_KT = 73728;      // K tile, 2 stages x 2 panels (dk 0-63, 64-127) x 64 token rows
// Rows 64-127 of the W S accumulator for the row sum, then U in place: fp32, 2 swizzled panels of 32
// columns x 64 rows (the TMA store's source for U)
constexpr uint32_t B_XCH = 106496;
constexpr uint32_t B_WG = 122880;     // W fp32 as 4 swizzled panels of 32 columns x 64 rows (32 KB), G [64], R [128]
constexpr uint32_t kWgStage = 33792, kWgG = 32768, kWgR = 33024;
constexpr uint32_t B_UT = B_WG + kWgStage;   // U~ of the slice, fp32, 2 swizzled panels of 32 columns x 64 rows
constexpr uint32_t B_SST = 174080;    // the next chunk-start state, fp32, 4 swizzled panels (rows 0-63 | 64-127 x 32 columns)
constexpr uint32_t B_BAR = B_SST + 32768;
constexpr uint32_t B_SMEM = B_BAR + 128 + 1024;
static_assert(B_SMEM <= 227 * 1024 && B_WG % 1024 == 0 && B_SST % 1024 == 0 && B_UT % 1024 == 0 && B_UT + 16384 <= B_SST &&
                  B_XCH + 16384 <= B_WG, "shared memory layout");
constexpr int kKStages = 2;
// 9 warps: warps 0-7 run the epilogues (warps w and w + 4 share TMEM lane quarter w % 4 and split
// the 64 columns); lane 0 of warp 8 issues the MMAs.
constexpr int kEpiThreads = 256, kThreads = kEpiThreads + 32, kIssuer = kEpiThreads;
// TMEM columns: [W_h; W_m] and [W_l; 0] as bf16 A operands, 64 columns each, 0-127 for even chunks
// and 128-255 for odd ones; W S accumulator 256-319; state S 320-383; K^T as the bf16 A operand
// 384-415.  The epilogue warps write K^T of a chunk and W of the next one while W S runs (an A
// operand from TMEM issues in about 58 cycles, an MN-major one from shared memory in about 137).
constexpr uint32_t T_AW = 0, T_D1 = 256, T_S = 320, T_AK = 384, kTmemCols = 512;

__device__ __forceinline__ void nb_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void nb_arrive(int id, int n) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// x = h + m + l (exact) in bf16 parts, each packed with its neighbour: lo holds x0's part, hi x1's.
__device__ __forceinline__ void split3(float x0, float x1, uint32_t& h, uint32_t& m, uint32_t& l) {
    constexpr uint32_t kHi = 0xffff0000u;
    const uint32_t h0 = __float_as_uint(x0) & kHi, h1 = __float_as_uint(x1) & kHi;
    const float r0 = x0 - __uint_as_float(h0), r1 = x1 - __uint_as_float(h1);
    const uint32_t m0 = __float_as_uint(r0) & kHi, m1 = __float_as_uint(r1) & kHi;
    const uint32_t l0 = __float_as_uint(r0 - __uint_as_float(m0)), l1 = __float_as_uint(r1 - __uint_as_float(m1));
    h = __byte_perm(h0, h1, 0x7632);   // upper halves: x0's part low, x1's high
    m = __byte_perm(m0, m1, 0x7632);
    l = __byte_perm(l0, l1, 0x7632);
}

// 32 fp32 values (consecutive columns of one row) -> the three bf16 parts, 16-byte chunks c0 .. c0 + 3
// of row r in the three panels at part0, part0 + pstride, part0 + 2 pstride (128-byte swizzle).
__device__ __forceinline__ void store_parts(uint8_t* part0, uint32_t pstride, int r, int c0, const uint32_t (&x)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t h[4], m[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            split3(__uint_as_float(x[8 * c + 2 * e]), __uint_as_float(x[8 * c + 2 * e + 1]), h[e], m[e], l[e]);
        const uint32_t o = swz((uint32_t)r, (uint32_t)(c0 + c));
        *reinterpret_cast<uint4*>(part0 + o) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(part0 + pstride + o) = make_uint4(m[0], m[1], m[2], m[3]);
        *reinterpret_cast<uint4*>(part0 + 2 * pstride + o) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
bwd_state_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_s,
                        const float* __restrict__ S0,
                        float* __restrict__ S_final, const float* __restrict__ ws_W, float* __restrict__ ws_U,
                        const float* __restrict__ ws_G, float* __restrict__ ws_S, const float* __restrict__ ws_R,
                        int T_len, int Hqk, int Hv, const int32_t* __restrict__ cu, int nseq, int normalize,
                        unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    // bar_w0: the W / G stage landed; bar_wfree: every epilogue warp has read it (count 8)
    const uint32_t bar_k0 = sb + B_BAR, bar_p1 = sb + B_BAR + 16, bar_p2 = sb + B_BAR + 24, bar_drain = sb + B_BAR + 32,
                   bar_w0 = sb + B_BAR + 40, bar_wfree = sb + B_BAR + 48, bar_ut = sb + B_BAR + 72;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + B_BAR + 56);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + B_BAR + 60);
    int* k_issued = reinterpret_cast<int*>(sm + B_BAR + 80);   // K tiles, W stages, U~ tiles issued

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp < kEpiThreads / 32;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int R = 32 * quarter + lane;   // TMEM lane: W S row (token R, or R - 64 for rows 64-127), S row (dk R)
    const int cb = 32 * half;            // this thread's 32 of the slice's 64 columns
    const int z = blockIdx.x % kSlices, h = (blockIdx.x / kSlices) % Hv, i = blockIdx.x / (kSlices * Hv);
    if (i >= nseq) return;
    const int hk = h / (Hv / Hqk), col0 = kSW * z;
    long long t0, t1;
    seq_range(cu, i, T_len, t0, t1);
    const long long nch = (t1 - t0 + kC - 1) / kC, slot0 = t0 / kC + i;

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tc_fence_before();
    }
    if (tid == 0) {
        *abort_flag = 0;
        k_issued[0] = k_issued[1] = k_issued[2] = 0;
        mbar_init(bar_ut, 1);
        for (int q = 0; q < kKStages; ++q) mbar_init(bar_k0 + 8 * q, 1);
        mbar_init(bar_w0, 1);
        mbar_init(bar_wfree, kEpiThreads / 32);
        mbar_init(bar_p1, 1);
        mbar_init(bar_p2, 1);
        mbar_fence_init();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);
    const size_t sbase = ((size_t)i * Hv + h) * kD * kD + col0;   // state slice of this CTA in S0 / S_final

    auto wi = [&](long long c) { return (size_t)(slot0 + c) * Hv + h; };
    auto wait_k = [&](long long c) {
        return mbar_wait_bounded(bar_k0 + 8 * (uint32_t)(c & 1), (uint32_t)((c >> 1) & 1), abort_flag, status,
                                 kStatusTimeout, kWaitLimitNs);
    };
    auto wait_group = [&](uint32_t bar, long long c) {
        return mbar_wait_bounded(bar, (uint32_t)(c & 1), abort_flag, status, kStatusTimeout, kWaitLimitNs);
    };
    bool waits_ok = true;   // a stage is refilled only by a thread whose own waits succeeded
    auto load_k = [&](long long c) {
        if (!waits_ok) return;
        const uint32_t st = (uint32_t)(c & 1), bar = bar_k0 + 8 * st;
        const int tc0 = (int)(t0 + c * kC);
        mbar_arrive_expect_tx(bar, 16384);
        tma_load_3d(sb + B_KT + st * 16384, &tm_k, 0, hk, tc0, bar);
        tma_load_3d(sb + B_KT + st * 16384 + 8192, &tm_k, 64, hk, tc0, bar);
        k_issued[0] = (int)(c + 1);
    };
    // one W / G stage: chunk c is its c-th load (phase c) and its c-th release (bar_wfree phase c)
    auto wait_w = [&](long long c) {
        return mbar_wait_bounded(bar_w0, (uint32_t)(c & 1), abort_flag, status, kStatusTimeout, kWaitLimitNs);
    };
    auto load_wg = [&](long long c) {   // W, G (and the row scalars) of chunk c into the stage
        if (!waits_ok) return;
        const uint32_t bar = bar_w0, dst = sb + B_WG;
        mbar_arrive_expect_tx(bar, kWgG + 256 + (normalize ? 512 : 0));
        for (int p = 0; p < 4; ++p)   // W rows of chunk c: rows wi(c) * 64 .. + 63 of the [rows, 128] fp32 view
            tma_load_2d(dst + p * 8192, &tm_w, 32 * p, (int)(wi(c) * kC), bar);
        bulk_g2s(dst + kWgG, ws_G + wi(c) * kC, 256, bar);
        if (normalize) bulk_g2s(dst + kWgR, ws_R + wi(c) * 2 * kC, 512, bar);
        k_issued[1] = (int)(c + 1);
    };
    auto wg_stage = [&](long long c) { (void)c; return reinterpret_cast<const float*>(sm + B_WG); };
    auto release_w = [&]() {   // this warp has read the W / G stage
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_wfree);
    };
    const uint64_t dSB = smem_desc(sb + B_SB, 1024, 1024), dUB = smem_desc(sb + B_UB, 1024, 1024);

    // ---- per-thread operand rows, loaded a chunk ahead
    const int wt = R & 63;   // W row of this thread (rows 64-127 of the stacked operand repeat the tokens)
    // [W_h; W_m] and [W_l; 0] rows of this lane of chunk c (its stage landed) into TMEM: 32 columns each,
    // K elements 64 half .. + 63
    auto put_w = [&](long long c) {
        const uint8_t* stage = reinterpret_cast<const uint8_t*>(wg_stage(c));
        uint32_t a1[32], a2[32];
#pragma unroll
        for (int e = 0; e < 16; ++e) {   // columns 64 half + 4 e .. + 3: panel 2 half + e / 8, 16-byte chunk e % 8
            const float4 x = *reinterpret_cast<const float4*>(stage + (2 * half + (e >> 3)) * 8192 + swz((uint32_t)wt, (uint32_t)(e & 7)));
            uint32_t hh, mm, ll;
            split3(x.x, x.y, hh, mm, ll);
            a1[2 * e] = R < 64 ? hh : mm;
            a2[2 * e] = R < 64 ? ll : 0u;
            split3(x.z, x.w, hh, mm, ll);
            a1[2 * e + 1] = R < 64 ? hh : mm;
            a2[2 * e + 1] = R < 64 ? ll : 0u;
        }
        const uint32_t aw = T_AW + 128 * (uint32_t)(c & 1);
        tmem_st32(tl + aw + 32 * half, a1);
        tmem_st32(tl + aw + 64 + 32 * half, a2);
    };
    // U~ of the slice of chunk c (its c-th load) by TMA, a chunk ahead
    const uint8_t* ut = sm + B_UT + half * 8192;   // panel of this thread's 32 columns
    auto load_u = [&](long long c) {
        if (!waits_ok) return;
        mbar_arrive_expect_tx(bar_ut, 16384);
        tma_load_2d(sb + B_UT, &tm_u, col0, (int)(wi(c) * kC), bar_ut);
        tma_load_2d(sb + B_UT + 8192, &tm_u, col0 + 32, (int)(wi(c) * kC), bar_ut);
        k_issued[2] = (int)(c + 1);
    };
    // K^T of chunk c into TMEM (the A operand of the state update): row R = dk R, tokens 32 half .. + 31
    auto put_k = [&](long long c) {
        const uint8_t* kt = sm + B_KT + (uint32_t)(c & 1) * 16384 + (R >> 6) * 8192;
        const uint32_t j = (uint32_t)((R & 63) >> 3), o = (uint32_t)(R & 7) * 2;
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const uint32_t t0 = (uint32_t)(32 * half + 2 * e), t1 = t0 + 1;
            const uint32_t lo = *reinterpret_cast<const uint16_t*>(kt + t0 * 128 + ((j ^ (t0 & 7)) << 4) + o);
            const uint32_t hi = *reinterpret_cast<const uint16_t*>(kt + t1 * 128 + ((j ^ (t1 & 7)) << 4) + o);
            w[e] = lo | (hi << 16);
        }
        tmem_st16(tl + T_AK + 16 * half, w);
    };
    auto row_b = [&](long long c) {   // b_R = exp(G_C - G_R) (/ |k_R|) of chunk c (stage landed), token rows R < 64
        const float* G = wg_stage(c) + kWgG / 4;
        const float rk = normalize ? wg_stage(c)[kWgR / 4 + R] : 1.f;
        return __expf(G[kC - 1] - G[R]) * rk;
    };
    auto gamma_c = [&](long long c) { return __expf(wg_stage(c)[kWgG / 4 + kC - 1]); };   // stage landed

    if (nch == 0) {   // empty sequence: the final state is the initial state
        if (S_final && epi) {
            for (int e = 0; e < 32; e += 4) {
                const size_t o = sbase + (size_t)R * kD + cb + e;
                *reinterpret_cast<float4*>(S_final + o) =
                    S0 ? *reinterpret_cast<const float4*>(S0 + o) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    } else {
        if (tid == kIssuer) {
            for (long long c = 0; c < kKStages && c < nch; ++c) load_k(c);
            load_wg(0);
            load_u(0);
        }
        float b_cur = 0.f, b_next = 0.f;
        if (epi) {   // prologue: S0 -> workspace, its parts -> SB, gamma_C(0) S0 -> TMEM; W(0) -> TMEM
            uint32_t v[32];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 x = S0 ? *reinterpret_cast<const float4*>(S0 + sbase + (size_t)R * kD + cb + e)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                v[e] = __float_as_uint(x.x); v[e + 1] = __float_as_uint(x.y);
                v[e + 2] = __float_as_uint(x.z); v[e + 3] = __float_as_uint(x.w);
                *reinterpret_cast<float4*>(ws_S + wi(0) * kD * kD + (size_t)R * kD + col0 + cb + e) = x;
            }
            store_parts(sm + B_SB, 16384, R, cb >> 3, v);
            waits_ok &= wait_w(0);
            const float g0 = gamma_c(0);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(g0 * __uint_as_float(v[e]));
            tmem_st32(tl + T_S + cb, v);
            put_w(0);
            if (R < 64) b_cur = row_b(0);
            release_w();
            tmem_wait_st();
        } else if (lane == 0 && nch > 1) {   // chunk 1's W once chunk 0's has been read
            waits_ok &= wait_group(bar_wfree, 0);
            load_wg(1);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        for (long long c = 0; c < nch; ++c) {
            const bool last = (c + 1 == nch);
            if (!epi) {   // ---- the issuing warp
                if (c > 0) nb_sync(1, kThreads);   // S_c parts in SB, gamma-scaled S_c and W_c in TMEM
                if (lane == 0) {   // D = [W_h; W_m] (S_h + S_m + S_l) + [W_l; 0] S_h
                    tc_fence_after();
                    const uint32_t aw = tmem + T_AW + 128 * (uint32_t)(c & 1);
#pragma unroll 1
                    for (int p = 0; p < 3; ++p)
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_bf16_ta(tmem + T_D1, aw + 8 * ks, dSB + ((p * 16384 + ks * 2048) >> 4),
                                        idesc_bf16(128, 64, 0, 1), (p > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ta(tmem + T_D1, aw + 64 + 8 * ks, dSB + ((ks * 2048) >> 4), idesc_bf16(128, 64, 0, 1), 1u);
                    mma_commit(bar_p1);
                    if (c + 2 < nch) {   // chunk c + 2's W once every warp has taken chunk c + 1's (this step's start)
                        waits_ok &= wait_group(bar_wfree, c + 1);
                        load_wg(c + 2);
                    }
                }
                __syncwarp();
                nb_sync(2, kThreads);   // the (bU) parts are in UB
                if (lane == 0) {   // S (gamma_C-scaled) += K^T ((bU)_h + (bU)_m + (bU)_l), K^T from TMEM
                    tc_fence_after();
#pragma unroll 1
                    for (int p = 0; p < 3; ++p)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16_ta(tmem + T_S, tmem + T_AK + 8 * ks, dUB + ((p * 8192 + ks * 2048) >> 4),
                                        idesc_bf16(128, 64, 0, 1), 1u);
                    mma_commit(bar_p2);
                    if (c + 2 < nch) load_k(c + 2);   // every warp has copied this chunk's K tile to TMEM
                }
                __syncwarp();
            } else {      // ---- the epilogue warps
                waits_ok &= wait_k(c);   // K^T of this chunk and W of the next into TMEM while W S runs
                put_k(c);
                float g_next = 1.f;
                if (!last) {   // (the previous chunk's W S, which read this W buffer, has completed)
                    waits_ok &= wait_w(c + 1);
                    put_w(c + 1);
                    g_next = gamma_c(c + 1);
                    if (R < 64) b_next = row_b(c + 1);
                    release_w();
                }
                waits_ok &= wait_group(bar_p1, c);
                tc_fence_after();
                {
                    uint32_t d[32];
                    tmem_ld32(tl + T_D1 + cb, d);
                    tmem_wait_ld();
                    uint8_t* xch = sm + B_XCH + half * 8192;   // panel of this thread's 32 columns
                    if (R >= 64) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(xch + swz((uint32_t)(R - 64), (uint32_t)(e >> 2))) =
                                make_float4(__uint_as_float(d[e]), __uint_as_float(d[e + 1]), __uint_as_float(d[e + 2]),
                                            __uint_as_float(d[e + 3]));
                    }
                    nb_sync(3, kEpiThreads);   // rows 64-127 of D are in shared memory
                    if (R < 64) {   // U = U~ - (D_r + D_{r+64}) to the workspace; b U as three parts into UB
                        waits_ok &= wait_group(bar_ut, c);
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            float4* xp = reinterpret_cast<float4*>(xch + swz((uint32_t)R, (uint32_t)(e >> 2)));
                            const float4 x = *xp;
                            const float4 y = *reinterpret_cast<const float4*>(ut + swz((uint32_t)R, (uint32_t)(e >> 2)));
                            const float4 u = make_float4(y.x - (__uint_as_float(d[e]) + x.x), y.y - (__uint_as_float(d[e + 1]) + x.y),
                                                         y.z - (__uint_as_float(d[e + 2]) + x.z), y.w - (__uint_as_float(d[e + 3]) + x.w));
                            *xp = u;   // U row R in place: the TMA store's source
                            d[e] = __float_as_uint(b_cur * u.x); d[e + 1] = __float_as_uint(b_cur * u.y);
                            d[e + 2] = __float_as_uint(b_cur * u.z); d[e + 3] = __float_as_uint(b_cur * u.w);
                        }
                        store_parts(sm + B_UB, 8192, R, cb >> 3, d);
                        fence_proxy_async_smem();
                        b_cur = b_next;
                        nb_sync(5, 128);            // every U row is in the exchange panels; U~ read
                        if (tid == 0) {             // U of chunk c to the workspace, U~ of chunk c + 1 in
                            tma_store_2d(&tm_u, col0, (int)(wi(c) * kC), sb + B_XCH);
                            tma_store_2d(&tm_u, col0 + 32, (int)(wi(c) * kC), sb + B_XCH + 8192);
                            bulk_commit();
                            if (!last) load_u(c + 1);
                        }
                    } else if (warp == 6 && lane == 0) {   // the previous state store has read its staging
                        bulk_wait_read();
                    }
                    tmem_wait_st();   // K^T is in TMEM
                    tc_fence_before();
                    nb_arrive(2, kThreads);
                }
                waits_ok &= wait_group(bar_p2, c);
                tc_fence_after();
                {   // new state row R: fp32 to the workspace (or S_final), parts into SB, gamma-scaled into TMEM
                    uint32_t vv[32];
                    tmem_ld32(tl + T_S + cb, vv);
                    tmem_wait_ld();
                    if (last && S_final) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4*>(S_final + sbase + (size_t)R * kD + cb + e) =
                                make_float4(__uint_as_float(vv[e]), __uint_as_float(vv[e + 1]), __uint_as_float(vv[e + 2]),
                                            __uint_as_float(vv[e + 3]));
                    }
                    if (!last) {
                        uint8_t* sst = sm + B_SST + ((R >> 6) * 2 + half) * 8192;   // panel (row half, column half)
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<uint4*>(sst + swz((uint32_t)(R & 63), (uint32_t)(e >> 2))) =
                                make_uint4(vv[e], vv[e + 1], vv[e + 2], vv[e + 3]);
                        store_parts(sm + B_SB, 16384, R, cb >> 3, vv);
#pragma unroll
                        for (int e = 0; e < 32; ++e) vv[e] = __float_as_uint(g_next * __uint_as_float(vv[e]));
                        tmem_st32(tl + T_S + cb, vv);
                        tmem_wait_st();
                        fence_proxy_async_smem();
                        tc_fence_before();
                        nb_sync(4, kEpiThreads);   // the state rows are in the staging panels
                        if (warp == 6 && lane == 0) {   // the chunk-start state of chunk c + 1 to the workspace
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                tma_store_2d(&tm_s, col0 + 32 * (q & 1), (int)(wi(c + 1) * kD + 64 * (q >> 1)),
                                             sb + B_SST + q * 8192);
                            bulk_commit();
                        }
                        if (tid == 0) bulk_wait_read();   // the U store has read the exchange panels
                        nb_arrive(1, kThreads);
                    }
                }
            }
        }
    }
    if (tid == 0 || (warp == 6 && lane == 0)) bulk_wait_all();   // TMA stores of U and S complete
    tc_fence_before();
    __syncthreads();
    if (tid == kIssuer && *abort_flag) {
        // A bounded wait gave up: every MMA has completed and no tile load is landing before the TMEM
        // and shared memory are released.
        mbar_init(bar_drain, 1);
        mbar_fence_init();
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0, kWaitLimitNs);
        const long long nk = k_issued[0], nw = k_issued[1], nu = k_issued[2];
        if (nu > 0) mbar_wait_drain(bar_ut, (uint32_t)((nu - 1) & 1), kWaitLimitNs);
        for (long long c = max(0LL, nk - kKStages); c < nk; ++c)
            mbar_wait_drain(bar_k0 + 8 * (uint32_t)(c & 1), (uint32_t)((c >> 1) & 1), kWaitLimitNs);
        if (nw > 0) mbar_wait_drain(bar_w0, (uint32_t)((nw - 1) & 1), kWaitLimitNs);
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ the adjoint chain
// Chunks in reverse, per (sequence, value head, 64-column slice); lam = dL/dS at a chunk's end (fp32,
// in TMEM), dO the output gradient, P = scale D o Q K^T (from the WY kernel):
//     dU  = b o (K lam) + P^T dO                       (to the workspace)
//     lam <- gamma_C lam + Q^T (s gamma o dO) - W^T dU  (the chunk-end values go to the workspace)
// with the same three-part splits: K lam = K (lam_h + lam_m + lam_l) and P^T dO = sum_p P^T_p dO
// (K, Q, dO exact bf16 inputs), Q^T (s gamma o dO) = sum_p Q^T (s gamma o dO)_p, and W^T dU over the
// six part pairs above 2^-22.  The 64-row products run as M = 128 MMAs whose rows 64-127 are not
// used.  Q^T, -W^T and P^T are written to TMEM by the epilogue warps as bf16 A operands (lane = the
// product's row) while K lam runs; the (s gamma o dO) parts are built by the warps of rows 64-127,
// which have no dU rows, into the lam parts' shared memory once K lam has read it.
constexpr uint32_t A_LB = 0;          // lam parts: MN-major B, 128 dk rows x 64 columns (16 KB each)
constexpr uint32_t A_UB = 49152;      // dU parts: MN-major B, 64 token rows x 64 columns (8 KB each)
constexpr uint32_t A_KT = 73728;      // K tile (2 panels x 64 token rows); K lam reads 64 rows past it
constexpr uint32_t A_QT = 90112;      // Q tile
constexpr uint32_t A_OT = 106496;     // dO slice, 2 stages x 64 token rows x 64 columns
constexpr uint32_t A_WST = 122880;    // W fp32, 4 swizzled panels of 32 columns x 64 rows
constexpr uint32_t A_PST = 155648;    // P fp32, 2 swizzled panels of 32 columns x 64 rows
constexpr uint32_t A_GST = 172032;    // G [64]
constexpr uint32_t A_XU = 173056;     // dU fp32, 2 swizzled panels (the TMA store's source)
constexpr uint32_t A_SST = 189440;    // a chunk-end lam, fp32, 4 swizzled panels (the TMA store's source)
constexpr uint32_t A_BAR = 222208;
constexpr uint32_t A_SMEM = A_BAR + 128 + 1024;
static_assert(A_SMEM <= 227 * 1024 && A_XU % 1024 == 0 && A_SST % 1024 == 0 && A_PST % 1024 == 0, "adjoint layout");
// TMEM: lam 0-63, K lam 64-127, P^T dO 128-191, Q^T 192-223, -W^T parts 288-383, P^T parts 384-479
// (32 columns a part: 64 K values).
constexpr uint32_t J_L = 0, J_D = 64, J_E = 128, J_AQ = 192, J_AW = 288, J_AP = 384;

__global__ void __launch_bounds__(kThreads, 1)
bwd_state_adj_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_du,
                        const __grid_constant__ CUtensorMap tm_ds, const float* __restrict__ ws_G,
                        const float* __restrict__ dS_final, float* __restrict__ grad_S0, float* __restrict__ ws_dS,
                        int T_len, int Hqk, int Hv, const int32_t* __restrict__ cu, int nseq, float scale,
                        unsigned* status, const float* __restrict__ ws_R, int normalize) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    // K tile, dO stages [2], staging (Q, W, P, G), K lam + P^T dO done, lam update done, drain
    const uint32_t bar_kt = sb + A_BAR, bar_o0 = sb + A_BAR + 8, bar_st = sb + A_BAR + 24, bar_du = sb + A_BAR + 32,
                   bar_l = sb + A_BAR + 40, bar_drain = sb + A_BAR + 48;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + A_BAR + 56);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + A_BAR + 60);
    int* issued = reinterpret_cast<int*>(sm + A_BAR + 64);   // K tiles, dO tiles, staging sets issued

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp < kEpiThreads / 32;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int R = 32 * quarter + lane, cb = 32 * half;
    const int z = blockIdx.x % kSlices, h = (blockIdx.x / kSlices) % Hv, i = blockIdx.x / (kSlices * Hv);
    if (i >= nseq) return;
    const int hk = h / (Hv / Hqk), col0 = kSW * z;
    long long t0, t1;
    seq_range(cu, i, T_len, t0, t1);
    const long long nch = (t1 - t0 + kC - 1) / kC, slot0 = t0 / kC + i;

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tc_fence_before();
    }
    if (tid == 0) {
        *abort_flag = 0;
        issued[0] = issued[1] = issued[2] = 0;
        mbar_init(bar_kt, 1);
        mbar_init(bar_o0, 1);
        mbar_init(bar_o0 + 8, 1);
        mbar_init(bar_st, 1);
        mbar_init(bar_du, 1);
        mbar_init(bar_l, 1);
        mbar_fence_init();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(32 * quarter) << 16);
    const size_t sbase = ((size_t)i * Hv + h) * kD * kD + col0;

    // chunks run c = nch - 1 .. 0; j = nch - 1 - c counts the steps (and each resource's loads)
    auto wi = [&](long long c) { return (size_t)(slot0 + c) * Hv + h; };
    auto wait_par = [&](uint32_t bar, uint32_t par) {
        return mbar_wait_bounded(bar, par, abort_flag, status, kStatusTimeout, kWaitLimitNs);
    };
    bool waits_ok = true;
    auto load_kt = [&](long long c) {
        if (!waits_ok) return;
        const int tc0 = (int)(t0 + c * kC);
        mbar_arrive_expect_tx(bar_kt, 16384);
        tma_load_3d(sb + A_KT, &tm_k, 0, hk, tc0, bar_kt);
        tma_load_3d(sb + A_KT + 8192, &tm_k, 64, hk, tc0, bar_kt);
        issued[0] += 1;
    };
    auto load_do = [&](long long c) {   // into stage (nch - 1 - c) & 1
        if (!waits_ok) return;
        const uint32_t st = (uint32_t)((nch - 1 - c) & 1), bar = bar_o0 + 8 * st;
        mbar_arrive_expect_tx(bar, 8192);
        tma_load_3d(sb + A_OT + st * 8192, &tm_do, col0, h, (int)(t0 + c * kC), bar);
        issued[1] += 1;
    };
    auto load_st = [&](long long c) {   // Q tile, W, P, G of chunk c
        if (!waits_ok) return;
        const int tc0 = (int)(t0 + c * kC);
        mbar_arrive_expect_tx(bar_st, 16384 + 32768 + 16384 + 256 + (normalize ? 512 : 0));
        tma_load_3d(sb + A_QT, &tm_q, 0, hk, tc0, bar_st);
        tma_load_3d(sb + A_QT + 8192, &tm_q, 64, hk, tc0, bar_st);
        for (int p = 0; p < 4; ++p) tma_load_2d(sb + A_WST + p * 8192, &tm_w, 32 * p, (int)(wi(c) * kC), bar_st);
        for (int p = 0; p < 2; ++p) tma_load_2d(sb + A_PST + p * 8192, &tm_p, 32 * p, (int)(wi(c) * kC), bar_st);
        bulk_g2s(sb + A_GST, ws_G + wi(c) * kC, 256, bar_st);
        // with in-kernel l2 normalisation: the rows' scalars 1/|k| (64) and 1/|q| (64) after G
        if (normalize) bulk_g2s(sb + A_GST + 256, ws_R + wi(c) * 2 * kC, 512, bar_st);
        issued[2] += 1;
    };
    const float* sG = reinterpret_cast<const float*>(sm + A_GST);
    const uint64_t dLB = smem_desc(sb + A_LB, 1024, 1024), dUB = smem_desc(sb + A_UB, 1024, 1024),
                   dKT = smem_desc(sb + A_KT, 16, 1024), dOT = smem_desc(sb + A_OT, 1024, 1024);

    // Q^T (exact), -W^T (rows = dk R, tokens 32 half .. + 31) and P^T (rows R < 64) of the staged chunk
    auto put_a = [&]() {
        uint32_t ph[16], pm[16], pl[16];
        const uint32_t jq = (uint32_t)((R & 63) >> 3), oq = (uint32_t)(R & 7) * 2;
#pragma unroll
        for (int e = 0; e < 16; ++e) {   // q_t[R], tokens t, t + 1
            const uint32_t ta = (uint32_t)(32 * half + 2 * e), tb = ta + 1;
            const uint8_t* qp = sm + A_QT + (R >> 6) * 8192;
            const uint32_t qa = *reinterpret_cast<const uint16_t*>(qp + ta * 128 + ((jq ^ (ta & 7)) << 4) + oq);
            const uint32_t qb = *reinterpret_cast<const uint16_t*>(qp + tb * 128 + ((jq ^ (tb & 7)) << 4) + oq);
            ph[e] = qa | (qb << 16);
        }
        tmem_st16(tl + J_AQ + 16 * half, ph);
        const uint32_t jw = (uint32_t)((R & 31) >> 2), ow = (uint32_t)(R & 3) * 4;
#pragma unroll
        for (int e = 0; e < 16; ++e) {   // -W[t][R]
            const uint32_t ta = (uint32_t)(32 * half + 2 * e), tb = ta + 1;
            const uint8_t* wp = sm + A_WST + (R >> 5) * 8192;
            const float wa = *reinterpret_cast<const float*>(wp + ta * 128 + ((jw ^ (ta & 7)) << 4) + ow);
            const float wb = *reinterpret_cast<const float*>(wp + tb * 128 + ((jw ^ (tb & 7)) << 4) + ow);
            split3(-wa, -wb, ph[e], pm[e], pl[e]);
        }
        tmem_st16(tl + J_AW + 16 * half, ph);
        tmem_st16(tl + J_AW + 32 + 16 * half, pm);
        tmem_st16(tl + J_AW + 64 + 16 * half, pl);
        if (R < 64) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {   // P[s][R], s = 32 half + 2 e, + 1
                const uint32_t sa = (uint32_t)(32 * half + 2 * e), sb2 = sa + 1;
                const uint8_t* pp = sm + A_PST + (R >> 5) * 8192;
                const float pa = *reinterpret_cast<const float*>(pp + sa * 128 + ((jw ^ (sa & 7)) << 4) + ow);
                const float pb = *reinterpret_cast<const float*>(pp + sb2 * 128 + ((jw ^ (sb2 & 7)) << 4) + ow);
                split3(pa, pb, ph[e], pm[e], pl[e]);
            }
            tmem_st16(tl + J_AP + 16 * half, ph);
            tmem_st16(tl + J_AP + 32 + 16 * half, pm);
            tmem_st16(tl + J_AP + 64 + 16 * half, pl);
        }
    };

    if (nch == 0) {   // no tokens: the gradient of S0 is that of S_final
        if (grad_S0 && epi) {
            for (int e = 0; e < 32; e += 4) {
                const size_t o = sbase + (size_t)R * kD + cb + e;
                *reinterpret_cast<float4*>(grad_S0 + o) =
                    dS_final ? *reinterpret_cast<const float4*>(dS_final + o) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    } else {
        if (tid == kIssuer) {
            load_kt(nch - 1);
            load_st(nch - 1);
            load_do(nch - 1);
            if (nch > 1) load_do(nch - 2);
        }
        if (epi) {   // lam of the last chunk's end: workspace, parts, gamma_C-scaled into TMEM
            uint32_t v[32];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 x = dS_final ? *reinterpret_cast<const float4*>(dS_final + sbase + (size_t)R * kD + cb + e)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                v[e] = __float_as_uint(x.x); v[e + 1] = __float_as_uint(x.y);
                v[e + 2] = __float_as_uint(x.z); v[e + 3] = __float_as_uint(x.w);
                *reinterpret_cast<float4*>(ws_dS + wi(nch - 1) * kD * kD + (size_t)R * kD + col0 + cb + e) = x;
            }
            store_parts(sm + A_LB, 16384, R, cb >> 3, v);
            waits_ok &= wait_par(bar_st, 0);
            const float g = __expf(sG[kC - 1]);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(g * __uint_as_float(v[e]));
            tmem_st32(tl + J_L + cb, v);
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        for (long long c = nch - 1; c >= 0; --c) {
            const long long j = nch - 1 - c;
            const uint32_t par = (uint32_t)(j & 1);
            if (!epi) {   // ---- the issuing warp
                if (j > 0) nb_sync(1, kThreads);   // lam parts in LB, gamma-scaled lam in TMEM
                if (lane == 0) {   // K lam = K (lam_h + lam_m + lam_l)
                    wait_par(bar_kt, par);
                    tc_fence_after();
#pragma unroll 1
                    for (int p = 0; p < 3; ++p)
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_bf16(tmem + J_D, dKT + (((ks >> 2) * 8192 + (ks & 3) * 32) >> 4),
                                     dLB + ((p * 16384 + ks * 2048) >> 4), idesc_bf16(128, 64, 0, 1), (p > 0 || ks > 0) ? 1u : 0u);
                }
                __syncwarp();
                nb_sync(2, kThreads);   // the A operands of this chunk are in TMEM; the staging was read
                if (lane == 0) {   // P^T dO, then lam += (s gamma o Q)^T dO
                    wait_par(bar_o0 + 8 * par, (uint32_t)((j >> 1) & 1));
                    tc_fence_after();
                    const uint64_t od = dOT + ((par * 8192u) >> 4);
#pragma unroll 1
                    for (int p = 0; p < 3; ++p)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16_ta(tmem + J_E, tmem + J_AP + 32 * p + 8 * ks, od + ((ks * 2048) >> 4),
                                        idesc_bf16(128, 64, 0, 1), (p > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(bar_du);
                    if (c > 0) load_st(c - 1);
                }
                __syncwarp();
                nb_sync(6, 160);   // the (s gamma o dO) parts are in the lam parts' shared memory
                if (lane == 0) {   // lam += Q^T (s gamma o dO)
                    tc_fence_after();
#pragma unroll 1
                    for (int p = 0; p < 3; ++p)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16_ta(tmem + J_L, tmem + J_AQ + 8 * ks, dLB + ((p * 8192 + ks * 2048) >> 4),
                                        idesc_bf16(128, 64, 0, 1), 1u);
                }
                __syncwarp();
                nb_sync(3, kThreads);   // the dU parts are in UB
                if (lane == 0) {   // lam -= W^T dU over the part pairs (h,h) (h,m) (m,h) (h,l) (l,h) (m,m)
                    tc_fence_after();
#pragma unroll 1
                    for (int q = 0; q < 6; ++q) {
                        const int a = (q == 2 || q == 5) ? 1 : (q == 4 ? 2 : 0);
                        const int u = (q == 1 || q == 5) ? 1 : (q == 3 ? 2 : 0);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16_ta(tmem + J_L, tmem + J_AW + 32 * a + 8 * ks, dUB + ((u * 8192 + ks * 2048) >> 4),
                                        idesc_bf16(128, 64, 0, 1), 1u);
                    }
                    mma_commit(bar_l);
                }
                __syncwarp();
            } else {      // ---- the epilogue warps
                float b = 0.f;   // rows R < 64: b_R; rows 64-127: s gamma of token R - 64 (0 past the sequence's end)
                const int n = (int)min((long long)kC, t1 - (t0 + c * kC));   // tokens of this chunk
                waits_ok &= wait_par(bar_st, par);   // this chunk's Q, W, P, G
                put_a();
                if (R < 64) b = __expf(sG[kC - 1] - sG[R]);
                else b = (R - 64) < n ? scale * __expf(sG[R - 64]) : 0.f;
                if (normalize) b *= sG[kC + R];   // K -> diag(1/|k|) K for rows R < 64, Q likewise for the rest
                tmem_wait_st();
                tc_fence_before();
                nb_arrive(2, kThreads);
                waits_ok &= wait_par(bar_du, par);
                tc_fence_after();
                if (warp == 7 && lane == 0 && c > 0) load_kt(c - 1);   // K lam has read the K tile
                if (R < 64) {   // dU = b o (K lam) + P^T dO: to the workspace and as three parts into UB
                    uint32_t d[32], e2[32];
                    tmem_ld32(tl + J_D + cb, d);
                    tmem_ld32(tl + J_E + cb, e2);
                    tmem_wait_ld();
                    uint8_t* xu = sm + A_XU + half * 8192;
                    const float bm = R < n ? b : 0.f, em = R < n ? 1.f : 0.f;   // rows past the sequence's end: 0
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        d[e] = __float_as_uint(fmaf(bm, __uint_as_float(d[e]), em * __uint_as_float(e2[e])));
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<uint4*>(xu + swz((uint32_t)R, (uint32_t)(e >> 2))) = make_uint4(d[e], d[e + 1], d[e + 2], d[e + 3]);
                    store_parts(sm + A_UB, 8192, R, cb >> 3, d);
                    fence_proxy_async_smem();
                    nb_sync(5, 128);
                    if (tid == 0) {
                        tma_store_2d(&tm_du, col0, (int)(wi(c) * kC), sb + A_XU);
                        tma_store_2d(&tm_du, col0 + 32, (int)(wi(c) * kC), sb + A_XU + 8192);
                        bulk_commit();
                    }
                } else {   // rows 64-127: (s gamma o dO) of token R - 64 as three parts (K lam has read LB)
                    const uint8_t* od = sm + A_OT + par * 8192;
                    const int t = R - 64;
                    uint32_t x[32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 u = *reinterpret_cast<const uint4*>(od + swz((uint32_t)t, (uint32_t)((cb >> 3) + q)));
                        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            x[8 * q + 2 * e] = __float_as_uint(b * __uint_as_float(w4[e] << 16));
                            x[8 * q + 2 * e + 1] = __float_as_uint(b * __uint_as_float(w4[e] & 0xffff0000u));
                        }
                    }
                    store_parts(sm + A_LB, 8192, t, cb >> 3, x);
                    fence_proxy_async_smem();
                    nb_arrive(6, 160);
                    if (warp == 6 && lane == 0) bulk_wait_read();   // the previous lam store has read its staging
                }
                tc_fence_before();
                nb_arrive(3, kThreads);
                waits_ok &= wait_par(bar_l, par);
                tc_fence_after();
                if (warp == 7 && lane == 0 && c >= 2) load_do(c - 2);   // this chunk's dO stage has been read
                {
                    uint32_t v[32];
                    tmem_ld32(tl + J_L + cb, v);
                    tmem_wait_ld();
                    if (c == 0) {   // lam at the first chunk's start: the gradient of S0
                        if (grad_S0) {
#pragma unroll
                            for (int e = 0; e < 32; e += 4)
                                *reinterpret_cast<float4*>(grad_S0 + sbase + (size_t)R * kD + cb + e) =
                                    make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                                __uint_as_float(v[e + 3]));
                        }
                    } else {   // lam at the end of chunk c - 1: workspace (TMA store), parts, gamma_C-scaled
                        uint8_t* sst = sm + A_SST + ((R >> 6) * 2 + half) * 8192;
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<uint4*>(sst + swz((uint32_t)(R & 63), (uint32_t)(e >> 2))) =
                                make_uint4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                        store_parts(sm + A_LB, 16384, R, cb >> 3, v);
                        waits_ok &= wait_par(bar_st, par ^ 1u);   // chunk c - 1's G
                        const float g = __expf(sG[kC - 1]);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(g * __uint_as_float(v[e]));
                        tmem_st32(tl + J_L + cb, v);
                        tmem_wait_st();
                        fence_proxy_async_smem();
                        tc_fence_before();
                        nb_sync(4, kEpiThreads);
                        if (warp == 6 && lane == 0) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                tma_store_2d(&tm_ds, col0 + 32 * (q & 1), (int)(wi(c - 1) * kD + 64 * (q >> 1)),
                                             sb + A_SST + q * 8192);
                            bulk_commit();
                        }
                        if (tid == 0) bulk_wait_read();   // the dU store has read its staging
                        nb_arrive(1, kThreads);
                    }
                }
            }
        }
    }
    if (tid == 0 || (warp == 6 && lane == 0)) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (tid == kIssuer && *abort_flag) {   // a bounded wait gave up: drain MMAs and loads before release
        mbar_init(bar_drain, 1);
        mbar_fence_init();
        mma_commit(bar_drain);
        mbar_wait_drain(bar_drain, 0, kWaitLimitNs);
        const int nk = issued[0], no = issued[1], ns = issued[2];
        if (nk > 0) mbar_wait_drain(bar_kt, (uint32_t)((nk - 1) & 1), kWaitLimitNs);
        if (ns > 0) mbar_wait_drain(bar_st, (uint32_t)((ns - 1) & 1), kWaitLimitNs);
        for (int q = max(0, no - 2); q < no; ++q)
            mbar_wait_drain(bar_o0 + 8 * (uint32_t)(q & 1), (uint32_t)((q >> 1) & 1), kWaitLimitNs);
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}
}  // namespace

cudaError_t launch_bwd_state_fwd_tc(const void* k, const float* S0, float* S_final, const float* ws_W, float* ws_U,
                                    const float* ws_G, float* ws_S, const float* ws_R, int T, int Hqk, int Hv,
                                    const int32_t* cu, int nseq, bool normalize, cudaStream_t stream,
                                    unsigned* status) {
    if ((reinterpret_cast<uintptr_t>(k) & 15u) != 0) return cudaErrorNotSupported;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (!encode) return cudaErrorNotSupported;
    const long long tokens = cu ? (long long)T : (long long)nseq * T;
    if (tokens > INT32_MAX) return cudaErrorInvalidValue;
    // k as [tokens, Hqk, 128] bf16, box of 64 features x 1 head x 64 tokens, 128-byte swizzle
    CUtensorMap tm;
    memset(&tm, 0, sizeof(tm));
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)Hqk, (cuuint64_t)(tokens > 0 ? tokens : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)Hqk * kD * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t elem[3] = {1, 1, 1};
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // W, U and S as 2-D fp32 tensors [rows, 128] (per chunk and head 64, 64 and 128 rows), boxes of 32
    // columns x 64 rows, 128-byte swizzle
    const long long slots = (tokens + kC - 1) / kC + nseq;
    if (slots * Hv * kD > INT32_MAX) return cudaErrorInvalidValue;
    auto map_f32 = [&](CUtensorMap* m, const float* base, long long rows) {
        memset(m, 0, sizeof(*m));
        const cuuint64_t d2[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
        const cuuint64_t s2[1] = {(cuuint64_t)kD * 4};
        const cuuint32_t b2[2] = {32, (cuuint32_t)kC};
        const cuuint32_t e2[2] = {1, 1};
        return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), d2, s2, b2, e2,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    CUtensorMap tw, tu, ts;
    if (!map_f32(&tw, ws_W, slots * Hv * kC) || !map_f32(&tu, ws_U, slots * Hv * kC) || !map_f32(&ts, ws_S, slots * Hv * kD))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(bwd_state_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)B_SMEM);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((long long)nseq * Hv * kSlices);
    bwd_state_fwd_tc_kernel<<<grid, kThreads, B_SMEM, stream>>>(tm, tw, tu, ts, S0, S_final, ws_W, ws_U, ws_G, ws_S, ws_R,
                                                                T, Hqk, Hv, cu, nseq, normalize ? 1 : 0, status);
    return cudaGetLastError();
}

}  // namespace gdn

namespace gdn {

cudaError_t launch_bwd_state_adj_tc(const void* q, const void* k, const void* dout, const float* dS_final,
                                    float* grad_S0, const float* ws_W, const float* ws_P, const float* ws_G,
                                    float* ws_dS, float* ws_dU, int T, int Hqk, int Hv, const int32_t* cu, int nseq,
                                    float scale, cudaStream_t stream, unsigned* status, const float* ws_R,
                                    bool normalize) {
    const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al16(q) || !al16(k) || !al16(dout)) return cudaErrorNotSupported;
    if (normalize && !ws_R) return cudaErrorInvalidValue;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (!encode) return cudaErrorNotSupported;
    const long long tokens = cu ? (long long)T : (long long)nseq * T;
    const long long slots = (tokens + kC - 1) / kC + nseq;
    if (tokens > INT32_MAX || slots * Hv * kD > INT32_MAX) return cudaErrorInvalidValue;
    // bf16 [tokens, heads, 128], boxes of 64 features x 1 head x 64 tokens; fp32 [rows, width], boxes of
    // 32 columns x 64 rows; 128-byte swizzle
    auto map_bf16 = [&](CUtensorMap* m, const void* base, int heads) {
        memset(m, 0, sizeof(*m));
        const cuuint64_t d3[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)(tokens > 0 ? tokens : 1)};
        const cuuint64_t s3[2] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2};
        const cuuint32_t b3[3] = {64, 1, 64};
        const cuuint32_t e3[3] = {1, 1, 1};
        return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), d3, s3, b3, e3,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    auto map_f32 = [&](CUtensorMap* m, const float* base, long long rows, int width) {
        memset(m, 0, sizeof(*m));
        const cuuint64_t d2[2] = {(cuuint64_t)width, (cuuint64_t)rows};
        const cuuint64_t s2[1] = {(cuuint64_t)width * 4};
        const cuuint32_t b2[2] = {32, (cuuint32_t)kC};
        const cuuint32_t e2[2] = {1, 1};
        return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), d2, s2, b2, e2,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    CUtensorMap tk, tq, to, tw, tp, tdu, tds;
    if (!map_bf16(&tk, k, Hqk) || !map_bf16(&tq, q, Hqk) || !map_bf16(&to, dout, Hv) ||
        !map_f32(&tw, ws_W, slots * Hv * kC, kD) || !map_f32(&tp, ws_P, slots * Hv * kC, kC) ||
        !map_f32(&tdu, ws_dU, slots * Hv * kC, kD) || !map_f32(&tds, ws_dS, slots * Hv * kD, kD))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(bwd_state_adj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)A_SMEM);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((long long)nseq * Hv * kSlices);
    bwd_state_adj_tc_kernel<<<grid, kThreads, A_SMEM, stream>>>(tk, tq, to, tw, tp, tdu, tds, ws_G, dS_final, grad_S0, ws_dS,
                                                                T, Hqk, Hv, cu, nseq, scale, status, ws_R, normalize ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace gdn
