// convert.cu -- FP16 <-> BF16 element copies, for FP16 inputs on the
// tensor-core path (whose MMAs take BF16 operands; one tcgen05 MMA cannot mix
// FP16 and BF16).  Each element is widened to FP32 exactly and rounded to
// the target type to nearest-even.  16-byte pieces when both pointers allow
// them, single elements for the rest.
#include "gdr_internal.cuh"

namespace gdr {
namespace {

template <typename Src, typename Dst>
__device__ __forceinline__ Dst cvt(Src x);
template <>
__device__ __forceinline__ __nv_bfloat16 cvt(__half x) {
    return __float2bfloat16_rn(__half2float(x));
}
template <>
__device__ __forceinline__ __half cvt(__nv_bfloat16 x) {
    return __float2half_rn(__bfloat162float(x));
}

template <typename Src, typename Dst>
__global__ void __launch_bounds__(256) k_convert(const Src *__restrict__ src, Dst *__restrict__ dst,
                                                 int64_t n, int vec) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t done = 0;
    if (vec) {  // eight elements per 16-byte piece
        const int64_t nv = n / 8;
        for (int64_t j = i; j < nv; j += stride) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(src) + j);
            const Src *s = reinterpret_cast<const Src *>(&raw);
            uint4 out;
            Dst *d = reinterpret_cast<Dst *>(&out);
#pragma unroll
            for (int e = 0; e < 8; ++e) d[e] = cvt<Src, Dst>(s[e]);
            reinterpret_cast<uint4 *>(dst)[j] = out;
        }
        done = nv * 8;
    }
    for (int64_t j = done + i; j < n; j += stride) dst[j] = cvt<Src, Dst>(src[j]);
}

template <typename Src, typename Dst>
cudaError_t launch_convert(const Src *src, Dst *dst, int64_t n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const int vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
    int64_t blocks = ((vec ? n / 8 : n) + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > 152 * 16) blocks = 152 * 16;
    k_convert<Src, Dst><<<(unsigned)blocks, 256, 0, st>>>(src, dst, n, vec);
    return cudaGetLastError();
}

}  // namespace

cudaError_t convert_f16_to_bf16(const void *src, void *dst, int64_t n, cudaStream_t st) {
    return launch_convert(static_cast<const __half *>(src), static_cast<__nv_bfloat16 *>(dst), n,
                          st);
}

cudaError_t convert_bf16_to_f16(const void *src, void *dst, int64_t n, cudaStream_t st) {
    return launch_convert(static_cast<const __nv_bfloat16 *>(src), static_cast<__half *>(dst), n,
                          st);
}

}  // namespace gdr
