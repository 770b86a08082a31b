// Declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedfp8.h"
#include "device.cuh"

namespace pkv {

constexpr int kHeadDim = PKV_HEAD_DIM;

// Decode kernel shape (shared by the launcher and the workspace sizing).
constexpr int kWarps = 4;                               // independent workers per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kCtasPerSm = 3;                           // resident decode CTAs per SM
constexpr int kPartialStride = kHeadDim + 4;            // floats per (slot, head): acc, m, l, pad

// Page sizes the library accepts (tokens per page).
inline bool page_size_ok(int p)
{
    return p == 16 || p == 32 || p == 64 || p == 128 || p == 256;
}

struct AppendArgs {
    const void *k_new, *v_new;
    int in_bf16;
    int64_t num_tokens;
    int hkv;
    const int64_t *slots;
    const float *k_scale, *v_scale;
    uint8_t *k_cache, *v_cache;
    int64_t num_pages;
    int page_size;
    int32_t *err;
};

// Longest chain of 16-token chunks one decode worker accumulates into one
// partial state: a worker whose range is longer cuts it into sub-pieces at
// every kChainChunks chunks of its range (the tensor cores' fp32 accumulation
// rounds toward zero, so error would otherwise grow with the chain).
constexpr int kChainChunks = 512;

// Decode workspace: a header, one record per (sequence, kv head) segment,
// then the partial-state slots.
struct DecodeHeader {
    long long total;                // chunk-heads in the list (all segments)
    int subs;                       // sub-pieces per worker range: ceil(ceil(total / workers) / kChainChunks)
    int pad;
};
struct SegRecord {
    long long start;                // list position of the segment's first chunk-head
    int n;                          // its chunks (0: empty sequence)
    int w0;                         // worker of its first chunk; -1: one piece, nothing to merge
};

struct DecodeArgs {
    const __nv_bfloat16 *q;
    const float *k_scale, *v_scale;
    const int32_t *block_table;
    int max_pages;
    const int32_t *seq_lens;
    int max_len;                    // bound of seq_lens (entries above are clamped and flagged)
    const int32_t *page_sizes;      // [batch] tokens per page of each sequence, or nullptr: all page_size
    int batch, hq, hkv, group;
    int page_size;                  // tokens per pool page (16..256); the kernel works in 16-token chunks
    int pool_log2;                  // log2(page_size)
    int64_t num_pages;
    float sm_scale_log2;        // sm_scale * log2(e): scores live in the exp2 domain
    void *out;
    int out_f32;
    // Fused append (pkv_append_decode_fp8): n_new new tokens per sequence at
    // positions seq_lens[b] - n_new .. seq_lens[b] - 1; k_new == nullptr: none.
    const void *k_new, *v_new;      // [batch][n_new][hkv][128], fp32 or bf16
    int new_bf16;
    int n_new;
    uint8_t *k_pool, *v_pool;       // the pools the tensor maps describe (for the stores)
    DecodeHeader *header;           // workspace header (written by CTA 0)
    SegRecord *segs;                // [batch * hkv] segment records (written by CTA 0)
    float *partials;                // [num_ctas * kWarps * subs + batch * hkv][group][kPartialStride]
    int32_t *err;
    int num_ctas;
    int withhold_worker;            // failure-detection test hook (-1 = off)
};

// Chunked prefill (csrc/prefill.cu).  The queries of all sequences are rows
// of q [total_q][hq][128]; sequence b owns rows cu_q[b] .. cu_q[b+1]-1, which
// sit at positions seq_lens[b] - n_b .. seq_lens[b] - 1.
struct PrefillArgs {
    const int32_t *cu_q;
    int total_q, max_q_len;
    int tokens_per_tile;            // 128 / group query tokens per CTA tile
    int max_tiles;                  // ceil(max_q_len / tokens_per_tile)
    const float *k_scale, *v_scale;
    const int32_t *block_table;
    int max_pages;
    const int32_t *seq_lens;
    int batch, hq, hkv, group;
    int page_size;
    int64_t num_pages;
    const uint8_t *k_cache, *v_cache;
    int max_kv_len;                 // bound of seq_lens; the 16-bit copies hold kv_pad rows per (sequence, kv head)
    int kv_pad;                     // max_kv_len rounded up to a key tile (128)
    __half *k16, *v16;              // 16-bit copies [batch * hkv][kv_pad][128] (caller workspace):
                                    // K as bf16 bits, V as f16, both exact widenings of E4M3
    int withhold_block;             // failure-detection test hook (-1 = off)
    float sm_scale_log2;
    void *out;
    int out_f32;
    int32_t *err;
};

// Workspace of pkv_paged_prefill: the 16-bit copies of K (bf16) and V (f16).
inline size_t prefill_workspace_bytes(int batch, int hkv, int max_kv_len)
{
    const size_t pad = (static_cast<size_t>(max_kv_len) + 127) / 128 * 128;
    return 2 * static_cast<size_t>(batch) * hkv * pad * 128 * sizeof(__half);
}

// Workspace = header + segment records (rounded to 256 bytes), then the
// partial slots.
inline size_t decode_segment_bytes(int batch, int hkv)
{
    return (sizeof(DecodeHeader) + static_cast<size_t>(batch) * hkv * sizeof(SegRecord) + 255) & ~size_t(255);
}

// Sub-pieces per worker range for a list of `total` chunk-heads over
// `workers` workers (at least 1).
inline __host__ __device__ long long decode_subs(long long total, long long workers)
{
    const long long per = (total + workers - 1) / workers;
    const long long s = (per + kChainChunks - 1) / kChainChunks;
    return s < 1 ? 1 : s;
}

// Host helpers (api.cu).
int device_sm_count();

// Launchers.
cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t stream);
cudaError_t launch_kv_calibrate(const void *k_new, const void *v_new, int in_bf16, int64_t T, int hkv,
                                float *k_max, float *v_max, float *k_scale, float *v_scale, cudaStream_t stream);
size_t decode_smem_bytes(int page_size, int batch);
const void *decode_kernel_for(int page_size);
int decode_num_ctas(int page_size, int batch, int max_ctas);
size_t decode_workspace_bytes(int batch, int hq, int hkv, long long max_len, int num_ctas);
size_t prefill_smem_bytes();
cudaError_t launch_paged_prefill(const PrefillArgs &a, const CUtensorMap &tm_q, const CUtensorMap &tm_k16,
                                 const CUtensorMap &tm_v16, cudaStream_t stream);
cudaError_t launch_paged_decode(const DecodeArgs &a, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                int page_size, cudaStream_t stream);

}  // namespace pkv
