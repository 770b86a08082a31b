// kv_calibrate: on-device KV-scale calibration.  Every attention layer keeps
// a running maximum of |K| and |V| per kv head over the prefill batches it has
// seen, and the FP8 scale used for every later token is that maximum / 448,
// floored at 1e-12 ("FP8量化与长上下文实测：Llama 3 70B部署优化指南", §3.2
// running max per layer, §3.1 absmax / 448 with clamp(min=1e-12)).
//
// Kernel 1 folds a batch of rows into the running maxima: each CTA reduces a
// token range of one (kv head, K or V) pair and merges its result with an
// integer atomicMax on the fp32 bits (exact: non-negative floats order like
// their bit patterns).  NaN values do not enter the maximum.  Kernel 2 turns
// the maxima into scales.
#include "internal.h"

namespace pkv {

namespace {

constexpr int kCalThreads = 256;

template <bool kBf16>
__global__ void __launch_bounds__(kCalThreads) kv_absmax_kernel(const void *__restrict__ k_new,
                                                                const void *__restrict__ v_new, int64_t T, int hkv,
                                                                int tokens_per_cta, float *__restrict__ k_max,
                                                                float *__restrict__ v_max)
{
    const int h = blockIdx.y;
    const bool is_v = blockIdx.z != 0;
    const void *x = is_v ? v_new : k_new;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * tokens_per_cta;
    const int64_t t1 = min(T, t0 + tokens_per_cta);
    float m = 0.f;
    // 16 dims per thread-step: rows of 128 dims are 8 chunks.
    for (int64_t c = t0 * 8 + threadIdx.x; c < t1 * 8; c += kCalThreads) {
        const int64_t t = c >> 3;
        const int part = static_cast<int>(c & 7);
        const int64_t e = (t * hkv + h) * kHeadDim + part * 16;
        if (kBf16) {
            const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(x) + e);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint4 u = __ldg(p + i);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    m = fmaxf(m, fabsf(__uint_as_float(w[k] << 16)));
                    m = fmaxf(m, fabsf(__uint_as_float(w[k] & 0xFFFF0000u)));
                }
            }
        } else {
            const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(x) + e);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = __ldg(p + i);
                m = fmaxf(fmaxf(m, fabsf(v.x)), fmaxf(fabsf(v.y), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float red[kCalThreads / 32];
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kCalThreads / 32; ++w)
            m = fmaxf(m, red[w]);
        atomicMax(reinterpret_cast<int *>((is_v ? v_max : k_max) + h), __float_as_int(m));
    }
}

__global__ void kv_scale_kernel(const float *__restrict__ k_max, const float *__restrict__ v_max, int hkv,
                                float *__restrict__ k_scale, float *__restrict__ v_scale)
{
    for (int i = threadIdx.x; i < 2 * hkv; i += blockDim.x) {
        const bool is_v = i >= hkv;
        const int h = is_v ? i - hkv : i;
        const float s = fmaxf(__fdiv_rn((is_v ? v_max : k_max)[h], 448.0f), 1e-12f);
        (is_v ? v_scale : k_scale)[h] = s;
    }
}

}  // namespace

cudaError_t launch_kv_calibrate(const void *k_new, const void *v_new, int in_bf16, int64_t T, int hkv,
                                float *k_max, float *v_max, float *k_scale, float *v_scale, cudaStream_t stream)
{
    if (T > 0) {
        const int sms = device_sm_count();
        int64_t ctas_x = (T + 63) / 64;
        const int64_t cap = (static_cast<int64_t>(sms) * 8 + 2 * hkv - 1) / (2 * hkv);
        if (ctas_x > cap)
            ctas_x = cap > 0 ? cap : 1;
        const int tokens_per_cta = static_cast<int>((T + ctas_x - 1) / ctas_x);
        const dim3 grid(static_cast<unsigned>(ctas_x), static_cast<unsigned>(hkv), 2);
        if (in_bf16)
            kv_absmax_kernel<true><<<grid, kCalThreads, 0, stream>>>(k_new, v_new, T, hkv, tokens_per_cta, k_max, v_max);
        else
            kv_absmax_kernel<false><<<grid, kCalThreads, 0, stream>>>(k_new, v_new, T, hkv, tokens_per_cta, k_max, v_max);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    if (k_scale && v_scale)
        kv_scale_kernel<<<1, 64, 0, stream>>>(k_max, v_max, hkv, k_scale, v_scale);
    return cudaGetLastError();
}

}  // namespace pkv

extern "C" pkv_status pkv_kv_calibrate(const void *k_new, const void *v_new, int in_dtype, int64_t num_tokens,
                                       int num_kv_heads, int head_dim, float *k_running_max, float *v_running_max,
                                       float *k_scale, float *v_scale, cudaStream_t stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || num_kv_heads > 65535)
        return PKV_ERR_SHAPE;
    if (in_dtype != PKV_F32 && in_dtype != PKV_BF16)
        return PKV_ERR_DTYPE;
    if (head_dim != pkv::kHeadDim)
        return PKV_ERR_UNSUPPORTED;
    if (!k_running_max || !v_running_max || (k_scale == nullptr) != (v_scale == nullptr))
        return PKV_ERR_NULL;
    if (num_tokens > 0 && (!k_new || !v_new))
        return PKV_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(k_new) & 15) || (reinterpret_cast<uintptr_t>(v_new) & 15) ||
        (reinterpret_cast<uintptr_t>(k_running_max) & 3) || (reinterpret_cast<uintptr_t>(v_running_max) & 3) ||
        (reinterpret_cast<uintptr_t>(k_scale) & 3) || (reinterpret_cast<uintptr_t>(v_scale) & 3))
        return PKV_ERR_ALIGN;
    return pkv::launch_kv_calibrate(k_new, v_new, in_dtype == PKV_BF16, num_tokens, num_kv_heads, k_running_max,
                                    v_running_max, k_scale, v_scale, stream) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}
