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

// Longest chain of 16-token chunks a decode worker accumulates on the tensor
// cores: every kFoldChunks chunks of a piece it adds its accumulator into the
// piece's partial-state slot in fp32 (round to nearest) and restarts it from
// zero (the tensor cores' fp32 accumulation rounds toward zero, so the error
// of one unbroken chain grows with its length).
constexpr int kFoldChunks = 128;
// Empty chunks the decode split counts after every segment (the cost of one
// more piece in a worker's range, two to three chunks' streaming time).
constexpr int kGhostChunks = 3;

// Weighted split.  Worker warp w = 4c + j of CTA c takes a share of the
// chunk-head list proportional to its CTA's weight (an integer in
// [kSplitWeightMin, kSplitWeightMax]; equal weights give the plain even split):
// with C(w) = 4 * sum_{c' < c} weight[c'] + j * weight[c] and CT = C(workers),
// worker w's range is [T * C(w) / CT, T * C(w + 1) / CT) (integer division).
// Weights are set per device for one grid size (a calibration measures how
// fast the SMs the CTAs land on stream their share); calls with another grid
// size split evenly.
constexpr int kMaxSplitCtas = 1024;
constexpr int kSplitWeightMin = 768;                   // weights are 1024 +- 25%, in steps of 1/1024
constexpr int kSplitWeightMax = 1280;

// Decode workspace: a header, one record per (sequence, kv head) segment,
// then the partial-state slots.
struct DecodeHeader {
    long long total;                // chunk-heads in the list (all segments)
    long long pad;
};
struct SegRecord {
    long long start;                // list position of the segment's first chunk-head
    int n;                          // its chunks (0: empty sequence)
    int w0;                         // worker of its first chunk; -1: one piece, nothing to merge
    int w1;                         // worker of its last chunk
    int pad;
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
    SegRecord *segs;                // [batch * hkv] segment records (written by the workers holding a
                                    // segment's first and last chunk)
    float *partials;                // [num_ctas * kWarps + batch * hkv][group][kPartialStride]: slot worker + list rank of the segment
    int32_t *err;
    int num_ctas;
    int withhold_worker;            // failure-detection test hook (-1 = off)
    // Split: split == 0 is the even split (CT = workers, every weight 1); else
    // the per-CTA weight prefix sums sit in device memory (see decode.cu) and
    // split_ct = C(workers), split_wmin / split_wmax bound the weights.
    int split;
    long long split_ct;
    int split_wmin, split_wmax;
    int probe;                      // calibration: record each CTA's start and end time
    long long num_slots;            // partial-state slots the workspace holds (accesses beyond: skipped, flagged)
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
    const int32_t *page_sizes;      // [batch] tokens per page of each sequence, or nullptr: all page_size
    int pool_log2;                  // log2(page_size)
    int max_kv_len;                 // bound of seq_lens
    int *tile_off;                  // [batch + 1] first 128-row tile of each sequence's widened region (caller
                                    // workspace, written by the widening kernel, read by the attention kernel)
    long long rows_cap;             // rows of the 16-bit copies the workspace holds
    __half *k16, *v16;              // 16-bit copies [rows_cap][128] (caller workspace): sequence b's kv head h
                                    // owns rows 128 * tile_off[b] + h * pad(L_b) .. + pad(L_b) - 1, pad = L
                                    // rounded up to 128; K as bf16 bits, V as f16, exact widenings of E4M3
    int withhold_block;             // failure-detection test hook (-1 = off)
    float sm_scale_log2;
    void *out;
    int out_f32;
    int32_t *err;
};

// Workspace of pkv_paged_prefill: the tile offsets of the sequences'
// regions (256-byte rounded), then the 16-bit copies of K (bf16) and of V
// (f16), each [rows][128].  Rows: the kv heads times the sum over sequences
// of L_b rounded up to 128, bounded by max_kv_len per sequence and, when
// given (> 0), by max_total_kv over the batch.
inline size_t prefill_header_bytes(int batch)
{
    return ((static_cast<size_t>(batch) + 1) * sizeof(int) + 255) & ~size_t(255);
}

inline long long prefill_rows_bound(int batch, int hkv, int max_kv_len, long long max_total_kv)
{
    long long tiles = static_cast<long long>(batch) * ((static_cast<long long>(max_kv_len) + 127) / 128);
    if (max_total_kv > 0) {
        const long long t2 = (max_total_kv + 127) / 128 + batch;   // sum of ceil(L_b / 128) <= sum L_b / 128 + batch
        tiles = t2 < tiles ? t2 : tiles;
    }
    return tiles * 128 * hkv;
}

inline size_t prefill_workspace_bytes(int batch, int hkv, int max_kv_len, long long max_total_kv)
{
    return prefill_header_bytes(batch) +
           2 * static_cast<size_t>(prefill_rows_bound(batch, hkv, max_kv_len, max_total_kv)) * 128 * sizeof(__half);
}

// Workspace = header + segment records (rounded to 256 bytes), then the
// partial slots.
inline size_t decode_segment_bytes(int batch, int hkv)
{
    return (sizeof(DecodeHeader) + static_cast<size_t>(batch) * hkv * sizeof(SegRecord) + 255) & ~size_t(255);
}

// ---------------------------------------------------------------- page walk
// Shared by decode and prefill (Args: DecodeArgs or PrefillArgs).  Sequence
// b's pages hold P_b tokens: a run of P_b / page_size consecutive pool pages
// whose first page is the block-table entry (P_b = page_size unless per-
// sequence page sizes are given).

// log2(P_b), or -1 if P_b is not a power of two in [page_size, 256].
template <typename Args>
__device__ __forceinline__ int seq_page_log2(const Args &a, int b)
{
    if (a.page_sizes == nullptr)
        return a.pool_log2;
    const int pb = __ldg(a.page_sizes + b);
    if (pb < a.page_size || pb > 256 || (pb & (pb - 1)) != 0)
        return -1;
    return 31 - __clz(pb);
}

// Pool page and row of token t of sequence b (lp = seq_page_log2): entry
// bt[b][t / P_b], offset o = t % P_b in pool page entry + o / page_size, row
// o % page_size.  False for an entry (or page) outside the pool.
template <typename Args>
__device__ __forceinline__ bool seq_token_page(const Args &a, int b, int lp, int t, int &phys, int &row)
{
    const int entry = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + (t >> lp));
    const int o = t & ((1 << lp) - 1);
    if (entry < 0 || entry >= a.num_pages)
        return false;
    phys = entry + (o >> a.pool_log2);
    row = o & (a.page_size - 1);
    return phys < a.num_pages;
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
                                int page_size, cudaStream_t stream, const char **site);
// Weighted split tables of the current device (decode.cu): the weight prefix
// sums (n + 1 entries) and the calibration's per-CTA [start, end] times.
cudaError_t upload_split_prefix(const uint32_t *prefix, int n);
cudaError_t clear_split_probe(int n, cudaStream_t stream);
cudaError_t read_split_probe(unsigned long long *times, int n);

}  // namespace pkv
