// Test-only: one tcgen05.mma kind::f16 product D[128 x N] = A[128 x K] B[K x N] with the operand
// layouts the prefill kernels use (128-byte-swizzled 64-column panels, K-major or MN-major), so a
// descriptor or layout mistake shows up on its own.  Operands are copied into shared memory with
// plain stores (in-bounds by construction: K <= 192, N <= 192), the product is read back from TMEM.
#include <cuda_bf16.h>
#include <stdint.h>

#include "tc_ptx.cuh"

using namespace gdn::tc;

namespace {

constexpr int kM = 128;

__global__ void __launch_bounds__(128, 1)
mma_case_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B, float* D, int K, int N, int a_mn, int b_mn,
                unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t A_OFF = 0, B_OFF = 49152, BAR = 49152 + 73728;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + BAR + 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + BAR + 12);
    const int tid = threadIdx.x, warp = tid >> 5;

    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tc_fence_before();
    }
    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(sb + BAR, 1);
        mbar_fence_init();
    }
    // A: K-major -> panels along K (128 rows x 64 cols); MN-major -> panels along M (K rows x 64 cols)
    for (int e = tid; e < kM * K; e += 128) {
        const int m = e / K, k = e % K;
        uint32_t off;
        if (!a_mn) off = (k / 64) * (kM * 128) + swz(m, (k % 64) / 8) + (k % 8) * 2;
        else off = (m / 64) * (K * 128) + swz(k, (m % 64) / 8) + (m % 8) * 2;
        *reinterpret_cast<__nv_bfloat16*>(sm + A_OFF + off) = A[e];
    }
    // B (logical K x N): K-major -> stored [N rows][K] panels along K; MN-major -> [K rows][N] panels along N
    for (int e = tid; e < K * N; e += 128) {
        const int k = e / N, n = e % N;
        uint32_t off;
        if (!b_mn) off = (k / 64) * (N * 128) + swz(n, (k % 64) / 8) + (k % 8) * 2;
        else off = (n / 64) * (K * 128) + swz(k, (n % 64) / 8) + (n % 8) * 2;
        *reinterpret_cast<__nv_bfloat16*>(sm + B_OFF + off) = B[e];
    }
    fence_proxy_async_smem();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) {
        for (int ks = 0; ks < K / 16; ++ks) {
            // MN-major: LBO = panel-to-panel offset along M/N (1024 when there is one panel only)
            const uint64_t ad = a_mn ? smem_desc(sb + A_OFF + ks * 2048, K * 128, 1024)
                                     : smem_desc(sb + A_OFF + (ks >> 2) * (kM * 128) + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = b_mn ? smem_desc(sb + B_OFF + ks * 2048, N > 64 ? K * 128 : 1024, 1024)
                                     : smem_desc(sb + B_OFF + (ks >> 2) * (N * 128) + (ks & 3) * 32, 16, 1024);
            mma_bf16(tmem, ad, bd, idesc_bf16(kM, N, a_mn, b_mn), ks > 0);
        }
        mma_commit(sb + BAR);
    }
    mbar_wait_bounded(sb + BAR, 0, abort_flag, status, 1u, 1000000000ull);
    tc_fence_after();
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    for (int cb = 0; cb < N / 32; ++cb) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * cb, r);
        tmem_wait_ld();
        for (int e = 0; e < 32; ++e) D[(size_t)tid * N + 32 * cb + e] = __uint_as_float(r[e]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

// A (128 x K, bf16) written into TMEM columns 128.. with tcgen05.st (lane m = row m, k pairs packed
// per 32-bit column, lower half = even k), B from shared memory (MN-major, or K-major when b_mn = 0),
// D into columns 0..N-1.
__global__ void __launch_bounds__(128, 1)
mma_tmem_a_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B, float* D, int K, int N, int b_mn,
                  unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t B_OFF = 0, BAR = 73728;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + BAR + 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + BAR + 12);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tc_fence_before();
    }
    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(sb + BAR, 1);
        mbar_fence_init();
    }
    for (int e = tid; e < K * N; e += 128) {
        const int k = e / N, n = e % N;
        const uint32_t off = b_mn ? (n / 64) * (K * 128) + swz(k, (n % 64) / 8) + (n % 8) * 2
                                  : (k / 64) * (N * 128) + swz(n, (k % 64) / 8) + (k % 8) * 2;
        *reinterpret_cast<__nv_bfloat16*>(sm + B_OFF + off) = B[e];
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    for (int cb = 0; cb < K / 64; ++cb) {   // row tid of A, k = 64 cb .. 64 cb + 63 -> 32 columns
        uint32_t v[32];
        for (int e = 0; e < 32; ++e) {
            const float lo = __bfloat162float(A[(size_t)tid * K + 64 * cb + 2 * e]);
            const float hi = __bfloat162float(A[(size_t)tid * K + 64 * cb + 2 * e + 1]);
            v[e] = pack_bf16(lo, hi);
        }
        tmem_st32(tl + 128 + 32 * cb, v);
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint64_t bd = b_mn ? smem_desc(sb + B_OFF + ks * 2048, N > 64 ? K * 128 : 1024, 1024)
                                     : smem_desc(sb + B_OFF + (ks >> 2) * (N * 128) + (ks & 3) * 32, 16, 1024);
            mma_bf16_ta(tmem, tmem + 128 + 8 * ks, bd, idesc_bf16(128, N, 0, b_mn), ks > 0);
        }
        mma_commit(sb + BAR);
    }
    mbar_wait_bounded(sb + BAR, 0, abort_flag, status, 1u, 1000000000ull);
    tc_fence_after();
    for (int cb = 0; cb < N / 32; ++cb) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * cb, r);
        tmem_wait_ld();
        for (int e = 0; e < 32; ++e) D[(size_t)tid * N + 32 * cb + e] = __uint_as_float(r[e]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

extern "C" int tc_selftest_mma_tmem_a(const void* A, const void* B, float* D, int K, int N, int b_mn,
                                      unsigned* status) {
    if (K % 64 || K < 64 || K > 128 || N % 64 || N < 64 || N > 128) return 1;
    const int smem = 73728 + 64 + 1024;
    if (cudaFuncSetAttribute(mma_tmem_a_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 2;
    mma_tmem_a_kernel<<<1, 128, smem>>>(static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B),
                                        D, K, N, b_mn, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int tc_selftest_mma(const void* A, const void* B, float* D, int K, int N, int a_mn, int b_mn,
                               unsigned* status) {
    if (K % 64 || K < 64 || K > 192 || N % 64 || N < 64 || N > 192) return 1;
    const int smem = 49152 + 73728 + 64 + 1024;
    if (cudaFuncSetAttribute(mma_case_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 2;
    mma_case_kernel<<<1, 128, smem>>>(static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), D,
                                      K, N, a_mn, b_mn, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// Failure detection without a fault: a wait on an mbarrier that nothing completes must give up after
// its limit, set the status flag and let the kernel return (the context stays usable).  One CTA;
// thread 0 waits, the others wait on the abort flag through the same bounded wait.
namespace {
__global__ void __launch_bounds__(64, 1) wait_runs_out_kernel(unsigned* status, unsigned long long limit_ns,
                                                              int* returned) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(b, 1);   // expects one arrival that never comes
        mbar_fence_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(b, 0, &abort_flag, status, 1u, limit_ns);
    __syncthreads();
    if (threadIdx.x == 0) *returned = ok ? 2 : 1;
}
}  // namespace

extern "C" int tc_selftest_wait_runs_out(unsigned* status, unsigned long long limit_ns, int* returned) {
    wait_runs_out_kernel<<<1, 64>>>(status, limit_ns, returned);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
