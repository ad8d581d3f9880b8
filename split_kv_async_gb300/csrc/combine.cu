// combine.cu -- cross-split combine: one CTA per softmax row (sequence b, query head h).
//
// opt.ai.kr "FlashDecoding++ async softmax -- theory", s3: with a unified max every split's
// partial (o_j, l_j) is already in the same frame, so only a plain sum remains. A split that
// was recomputed with online softmax carries its own max m_j, so the general form is
//     M = max_j m_j,  out = sum_j w_j o_j / sum_j w_j l_j,  w_j = exp(m_j - M)
// with w_j = 1 exactly when m_j == M: if no split of the row fell back (all m_j = phi) this is
// exactly the plain sum. Splits are summed in ascending j (deterministic), in fp32; the result
// is rounded to nearest even into the output dtype.
#include <cuda_bf16.h>

#include "device_common.cuh"

namespace fdpp {
namespace {

template <typename T>
__device__ __forceinline__ void store_out(T* p, float x);

template <>
__device__ __forceinline__ void store_out<float>(float* p, float x) { *p = x; }

template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float x)
{
    *p = __float2bfloat16_rn(x);
}

template <typename T>
__global__ void __launch_bounds__(128) combine_kernel(KernelArgs a)
{
    const int row = blockIdx.x;             // b * Hq + h
    const int b = row / a.Hq;
    const int n = a.nsplit[b];
    const long long base = (long long)row * a.max_splits;
    const float* m = a.m_part + base;
    const float* l = a.l_part + base;
    const float* o = a.o_part + base * a.D;
    T* out = static_cast<T*>(a.out) + (long long)row * a.D;

    float M = -INFINITY;
    for (int j = 0; j < n; ++j) M = fmaxf(M, m[j]);
    for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
        float acc = 0.f, lam = 0.f;
        for (int j = 0; j < n; ++j) {
            const float w = frame_weight(m[j], M);
            acc = fmaf(w, o[(long long)j * a.D + d], acc);
            lam = fmaf(w, l[j], lam);
        }
        store_out<T>(out + d, n > 0 ? __fdiv_rn(acc, lam) : 0.f);
    }
}

}  // namespace

cudaError_t launch_combine(const KernelArgs& a, int dtype, cudaStream_t s)
{
    const int rows = a.B * a.Hq;
    const int threads = a.D;
    if (dtype == FDPP_F32)
        combine_kernel<float><<<rows, threads, 0, s>>>(a);
    else
        combine_kernel<__nv_bfloat16><<<rows, threads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace fdpp
