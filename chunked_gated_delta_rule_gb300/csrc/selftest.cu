// selftest.cu -- diagnostic kernels that check, on the GPU, the tensor-core
// building blocks the fused path relies on: every operand layout of the
// tcgen05 MMA it issues (K-major and MN-major, 128-byte swizzle, M = 128,
// N = 64 / 128, K = 64 / 128) and the TMA tile load with 128-byte swizzle
// decoded through sw128_off.  Tests compare their results with PyTorch.
#include "gdr_internal.cuh"
#include "gdr_selftest.h"
#include "tc_common.cuh"
#include "tc_inverse.cuh"
#include "tma_host.cuh"

namespace gdr {
namespace {

using namespace tc;

// D[128][N] = A[128][Kd] * B[N][Kd]^T with A, B staged by threads into the
// requested layouts (a_mn = 2: A in tensor memory, packed two BF16 per
// column), one tcgen05.mma per 16-wide K step, FP32 in TMEM.
__global__ void __launch_bounds__(128)
k_selftest_umma(const __nv_bfloat16 *__restrict__ A, const __nv_bfloat16 *__restrict__ B,
                float *__restrict__ D, int N, int Kd, int a_mn, int b_mn, int32_t *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = base;
    uint8_t *sB = sA + 128 * Kd * 2;
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5;

    if (a_mn != 2) {
        for (int idx = tid; idx < 128 * Kd; idx += 128) {
            const int m = idx / Kd, k = idx - m * Kd;
            const uint32_t off = a_mn ? sw128_off(k, m, Kd) : sw128_off(m, k, 128);
            *reinterpret_cast<__nv_bfloat16 *>(sA + off) = A[idx];
        }
    }
    for (int idx = tid; idx < N * Kd; idx += 128) {
        const int n = idx / Kd, k = idx - n * Kd;
        const uint32_t off = b_mn ? sw128_off(k, n, Kd) : sw128_off(n, k, N);
        *reinterpret_cast<__nv_bfloat16 *>(sB + off) = B[idx];
    }
    fence_async_smem();
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    const uint32_t dcol = a_mn == 2 ? 128u : 0u;  // D after A when A is in TMEM
    if (a_mn == 2) {  // row tid of A, packed, into columns [0, Kd / 2)
        for (int c0 = 0; c0 < Kd / 2; c0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const __nv_bfloat16 lo = A[tid * Kd + 2 * (c0 + i)];
                const __nv_bfloat16 hi = A[tid * Kd + 2 * (c0 + i) + 1];
                r[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
            }
            tmem_st32(tmem_addr(tbase, 32 * warp, c0), r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(128, N, a_mn == 1, b_mn);
        for (int kk = 0; kk < Kd / 16; ++kk) {
            const int k0 = kk * 16;
            uint64_t ad = 0, bd;
            if (a_mn == 0)
                ad = sdesc_sw128(smem_u32(sA) + (k0 / 64) * 128 * 128 + (k0 % 64) * 2, 16, 1024);
            else if (a_mn == 1)
                ad = sdesc_sw128(smem_u32(sA) + k0 * 128, Kd * 128, 1024);
            if (!b_mn)
                bd = sdesc_sw128(smem_u32(sB) + (k0 / 64) * N * 128 + (k0 % 64) * 2, 16, 1024);
            else
                bd = sdesc_sw128(smem_u32(sB) + k0 * 128, Kd * 128, 1024);
            if (a_mn == 2)
                umma_bf16_ts(tbase + dcol, tbase + (uint32_t)(k0 / 2), bd, idesc, kk > 0 ? 1u : 0u);
            else
                umma_bf16(tbase, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bar);
    }
    __syncwarp();
    const bool ok = mbar_wait(&bar, 0, status);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            float f[16];
            tmem_load16f(tmem_addr(tbase, 32 * warp, dcol + c0), f);
#pragma unroll
            for (int i = 0; i < 16; ++i) D[tid * N + c0 + i] = f[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

// One 64 x 64 BF16 box of a [T][H][K] tensor at (t0, h, k0), loaded by TMA
// with 128-byte swizzle and read back element by element via sw128_off.
__global__ void __launch_bounds__(128)
k_selftest_tma(const __grid_constant__ CUtensorMap map, __nv_bfloat16 *__restrict__ out,
               int t0, int h, int k0, int32_t *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tile = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar;
    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar, 64 * 128);
        tma_load_3d(tile, &map, &bar, k0, h, t0);
    }
    const bool ok = mbar_wait(&bar, 0, status);
    if (!ok) return;
    for (int idx = tid; idx < 64 * 64; idx += 128) {
        const int r = idx >> 6, c = idx & 63;
        out[idx] = *reinterpret_cast<const __nv_bfloat16 *>(tile + sw128_off(r, c, 64));
    }
}

// T = (I + A)^-1 for one strictly lower 64 x 64 FP32 matrix, through the same
// device routine the tensor-core chain kernel uses.
__global__ void __launch_bounds__(256) k_selftest_inverse(const float *__restrict__ A,
                                                          float *__restrict__ T) {
    __shared__ float sAT[64 * kInvLd];
    __shared__ float sX[kInvScratchFloats];
    const int tid = threadIdx.x;
    for (int idx = tid; idx < 64 * 64; idx += 256) {
        const int i = idx >> 6, j = idx & 63;
        sAT[i * kInvLd + j] = j < i ? A[idx] : 0.f;
    }
    __syncthreads();
    invert_unit_lower64(sAT, sX, tid);
    for (int idx = tid; idx < 64 * 64; idx += 256) {
        const int i = idx >> 6, j = idx & 63;
        T[idx] = j <= i ? sAT[i * kInvLd + j] : 0.f;
    }
}

// Waits on an mbarrier that nothing completes, with a time limit: the wait
// must give up, record GDR_ERR_TIMEOUT in the status word and let the kernel
// finish normally (the failure path of every bounded wait in the library).
__global__ void k_selftest_timeout(int32_t *status, uint64_t limit_ns, int32_t *done) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, status, limit_ns);
    if (threadIdx.x == 0) *done = ok ? 1 : 2;
}

}  // namespace
}  // namespace gdr

using namespace gdr;

extern "C" int gdr_selftest_timeout(int32_t *status, uint64_t limit_ns, int32_t *done,
                                    gdr_stream_t stream) {
    if (!status || !done || limit_ns == 0 || limit_ns > 100000000ull) return GDR_ERR_INVALID;
    k_selftest_timeout<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status, limit_ns,
                                                                            done);
    return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

extern "C" int gdr_selftest_inverse(const float *A, float *T, gdr_stream_t stream) {
    if (!A || !T) return GDR_ERR_INVALID;
    k_selftest_inverse<<<1, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(A, T);
    return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

extern "C" int gdr_selftest_umma(const void *A, const void *B, float *D, int N, int Kd,
                                 int a_mn, int b_mn, int32_t *status, gdr_stream_t stream) {
    if (!A || !B || !D) return GDR_ERR_INVALID;
    if ((N != 64 && N != 128) || (Kd != 64 && Kd != 128) || a_mn < 0 || a_mn > 2 || (b_mn & ~1))
        return GDR_ERR_INVALID;
    const size_t smem = 1024 + (size_t)(128 + N) * Kd * 2;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaFuncSetAttribute(k_selftest_umma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return GDR_ERR_CUDA;
    k_selftest_umma<<<1, 128, smem, st>>>(static_cast<const __nv_bfloat16 *>(A),
                                          static_cast<const __nv_bfloat16 *>(B), D, N, Kd,
                                          a_mn, b_mn, status);
    return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

extern "C" int gdr_selftest_tma(const void *src, int64_t T, int64_t H, int64_t K, int t0, int h,
                                int k0, void *out, int32_t *status, gdr_stream_t stream) {
    if (!src || !out || T < 1 || H < 1 || K < 64 || K % 8) return GDR_ERR_INVALID;
    if (k0 % 8 || k0 < 0 || k0 + 64 > K || h < 0 || h >= H) return GDR_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(src) % 16) return GDR_ERR_INVALID;
    CUtensorMap map;
    if (!make_tmap_bf16_3d(&map, src, (uint64_t)K, (uint64_t)H, (uint64_t)T, (uint64_t)K * 2,
                           (uint64_t)H * K * 2, 64, 1, 64))
        return GDR_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    k_selftest_tma<<<1, 128, 1024 + 64 * 128, st>>>(map, static_cast<__nv_bfloat16 *>(out), t0, h, k0, status);
    return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}
