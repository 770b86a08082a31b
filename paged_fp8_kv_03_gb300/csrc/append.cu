// kv_append_fp8: quantise new K/V rows to E4M3 and scatter them into pages.
//
// Quantisation is a division by the per-head scale followed by the cast to
// E4M3 ("FP8量化与长上下文实测：Llama 3 70B部署优化指南", §3.1 weight recipe,
// §3.2 the same per-layer scale applied to new KV during decode); the cast
// rounds to nearest even and saturates at +-448 (§1.1 range).  Pages of P
// tokens, one block-table entry per page (0539edu.com Llama 3 notes, §2.2).
//
// One thread owns one 16-dim chunk of one (token, kv head) row for both K and
// V: 64 B (fp32) or 32 B (bf16) of coalesced input per tensor, one 16-byte
// store per tensor into the page row.
#include "internal.h"

namespace pkv {

namespace {

template <bool kBf16>
__device__ __forceinline__ void load16(const void *base, int64_t elem, float (&x)[16])
{
    if (kBf16) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(base) + elem);
        uint4 u[2] = {__ldg(p), __ldg(p + 1)};
        const uint32_t *w = reinterpret_cast<const uint32_t *>(u);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + elem);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 v = __ldg(p + i);
            x[4 * i] = v.x;
            x[4 * i + 1] = v.y;
            x[4 * i + 2] = v.z;
            x[4 * i + 3] = v.w;
        }
    }
}

// 16 values / scale (IEEE division) -> 16 E4M3 bytes (RNE, saturating).
__device__ __forceinline__ uint4 quantise16(const float (&x)[16], float scale)
{
    return make_uint4(quantise4(x[0], x[1], x[2], x[3], scale), quantise4(x[4], x[5], x[6], x[7], scale),
                      quantise4(x[8], x[9], x[10], x[11], scale), quantise4(x[12], x[13], x[14], x[15], scale));
}

template <bool kBf16>
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(
    const void *__restrict__ k_new, const void *__restrict__ v_new, int64_t num_tokens, int hkv,
    const int64_t *__restrict__ slot_mapping, const float *__restrict__ k_scale,
    const float *__restrict__ v_scale, uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
    int64_t num_slots, int page_size, int32_t *__restrict__ err)
{
    constexpr int kChunks = kHeadDim / 16;
    const int64_t total = num_tokens * hkv * kChunks;
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < total;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int part = static_cast<int>(c % kChunks);
        const int64_t row = c / kChunks;            // token * hkv + head
        const int h = static_cast<int>(row % hkv);
        const int64_t t = row / hkv;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            if (err && part == 0)
                atomicOr(err, PKV_DEVERR_SLOT);
            continue;
        }
        const int64_t page = slot / page_size;
        const int64_t off = slot - page * page_size;
        const int64_t src = row * kHeadDim + part * 16;
        const int64_t dst = ((page * hkv + h) * page_size + off) * kHeadDim + part * 16;
        float x[16];
        load16<kBf16>(k_new, src, x);
        *reinterpret_cast<uint4 *>(k_cache + dst) = quantise16(x, __ldg(k_scale + h));
        load16<kBf16>(v_new, src, x);
        *reinterpret_cast<uint4 *>(v_cache + dst) = quantise16(x, __ldg(v_scale + h));
    }
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t stream)
{
    const int64_t total = a.num_tokens * a.hkv * (kHeadDim / 16);
    if (total == 0)
        return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (blocks > cap)
        blocks = cap;
    const int64_t num_slots = a.num_pages * a.page_size;
    if (a.in_bf16)
        kv_append_fp8_kernel<true><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            a.k_new, a.v_new, a.num_tokens, a.hkv, a.slots, a.k_scale, a.v_scale, a.k_cache,
            a.v_cache, num_slots, a.page_size, a.err);
    else
        kv_append_fp8_kernel<false><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            a.k_new, a.v_new, a.num_tokens, a.hkv, a.slots, a.k_scale, a.v_scale, a.k_cache,
            a.v_cache, num_slots, a.page_size, a.err);
    return cudaGetLastError();
}

}  // namespace pkv
