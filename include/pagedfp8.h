/*
 * pagedfp8 -- paged FP8 (E4M3) KV cache and grouped-query decode attention
 * for sm_103a (GB300).  Plain C ABI: device pointers, sizes, a CUDA stream.
 *
 * Sources for what the calls compute (prior art; no kernel API is given
 * there):
 *   [G]  "FP8量化与长上下文实测：Llama 3 70B部署优化指南" (sheratonhq.com/news/163163):
 *        §1.1 the E4M3 format (max 448, smallest step 2^-9); §1.2 GQA, 8 KV
 *        heads serving 64 query heads, and quantising the KV cache to FP8;
 *        §2.2 the KV size 2 x layers x kv_heads x head_dim x tokens x bytes;
 *        §3.1 quantisation as a division by an absmax/448 scale; §3.2 one KV
 *        scale per attention layer, applied to every new K/V during decode.
 *   [N]  Llama 3 FP8 + 128K production notes (0539edu.com/news/5628500):
 *        §2.2 PagedAttention keeps the KV cache in fixed 16-token pages;
 *        §3.2 decode at 128K re-reads the whole cache every step, so it is
 *        bound by memory bandwidth; §3.3 block_size 16, kv_cache_dtype fp8;
 *        §5.2 one block-table entry per 16 tokens (8000 for 128000 tokens).
 *   [S]  Llama 3 8B notes (mlqm.cn/news/162512), §3.3: block size 32 option.
 *   [T]  Llama 3 technical notes (wmrh.cn/news/61679), §3.2: 256-token pages.
 *        [N] §3.2 also proposes 64-token pages for long segments.
 *
 * Memory layout (part of the ABI, so page bytes compare bit for bit):
 *   k_cache, v_cache : uint8  [num_pages][num_kv_heads][page_size][head_dim]
 *                      one pair per layer; a page holds page_size tokens of
 *                      every kv head, each kv head's tokens contiguous.
 *   block_table      : int32  [batch][max_pages_per_seq]; entry p of row b is
 *                      the physical page holding tokens p*P .. p*P+P-1.
 *   slot             : physical_page * page_size + row within the page.
 *
 * Ownership: the caller owns every buffer (caches, tables, outputs, the
 * decode workspace).  The library allocates no device memory, keeps no state
 * between calls beyond a per-device cache of device properties, the driver
 * entry point it uses to describe tensors for the TMA unit and the optional
 * per-device split weights (pkv_decode_set_split_weights), and never
 * synchronises the stream.  Calls are asynchronous on `stream`; the status
 * reports argument errors found on the host and launch errors only
 * (pkv_last_cuda_error names the CUDA error behind a PKV_ERR_CUDA).
 *
 * Device-side error word: kernels OR bits into *device_error (int32, device
 * memory, may be NULL) instead of reading or writing out of bounds:
 *   PKV_DEVERR_SLOT      a slot outside the pool (token skipped)
 *   PKV_DEVERR_PAGE      a block-table entry outside [0, num_pages) (its
 *                        page is read as zeros)
 *   PKV_DEVERR_SEQLEN    seq_lens[b] < 0, beyond max_seq_len or beyond
 *                        max_pages_per_seq pages (clamped)
 *   PKV_DEVERR_TIMEOUT   a pipeline wait exceeded its time limit (the kernel
 *                        stopped issuing work, drained its copies and
 *                        returned; outputs are undefined)
 *   PKV_DEVERR_PAGESIZE  a per-sequence page size that is not a power of two
 *                        in [page_size, 256] (the sequence is treated as
 *                        empty: zero output rows)
 *   PKV_DEVERR_INTERNAL  the decode's own split-K bookkeeping pointed outside
 *                        the workspace (the access was skipped; outputs are
 *                        not valid; not expected to happen)
 * The word is sticky: clear it (pkv_read_device_error with clear = 1, or
 * cudaMemsetAsync) before a call whose errors you want to attribute.
 */
#ifndef PAGEDFP8_H
#define PAGEDFP8_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int pkv_status;

enum {
    PKV_OK = 0,
    PKV_ERR_NULL = 1,         /* a required pointer is NULL                  */
    PKV_ERR_SHAPE = 2,        /* a size is negative, zero or inconsistent     */
    PKV_ERR_DTYPE = 3,        /* unknown dtype code                           */
    PKV_ERR_UNSUPPORTED = 4,  /* valid but not built: head_dim, page size, G  */
    PKV_ERR_WORKSPACE = 5,    /* workspace too small or misaligned            */
    PKV_ERR_CUDA = 6,         /* a CUDA runtime/driver call or launch failed  */
    PKV_ERR_ALIGN = 7         /* a pointer is not 16-byte aligned             */
};

/* Activation dtype codes. */
enum { PKV_F32 = 0, PKV_BF16 = 1 };

/* Device error bits (see above). */
enum {
    PKV_DEVERR_SLOT = 1,
    PKV_DEVERR_PAGE = 2,
    PKV_DEVERR_SEQLEN = 4,
    PKV_DEVERR_TIMEOUT = 8,
    PKV_DEVERR_PAGESIZE = 16,
    PKV_DEVERR_INTERNAL = 32
};

/* Build limits. */
#define PKV_HEAD_DIM 128      /* the only head_dim built (Llama 3)            */
#define PKV_MAX_GROUP 8       /* query heads per kv head, 1..8                */
#define PKV_MAX_BATCH 8192    /* sequences per decode call                    */

/*
 * kv_append_fp8 -- quantise new K and V tokens to E4M3 and write them into
 * their pages ([G] §3.1/§3.2 quantisation by division by the scale; [G] §1.1
 * format; [N] §2.2 pages).
 *
 * For every token t < num_tokens with slot = slot_mapping[t] >= 0, every kv
 * head h and every d < head_dim:
 *     k_cache[slot / P][h][slot % P][d] = E4M3(k_new[t][h][d] / k_scale[h])
 * and the same for V.  The division is IEEE fp32 (correctly rounded); E4M3 is
 * round-to-nearest-even from fp32 with saturation to +-448 (+-Inf -> +-448,
 * NaN -> a NaN code).
 *
 *   k_new, v_new   device, [num_tokens][num_kv_heads][head_dim], contiguous,
 *                  dtype in_dtype (PKV_F32 or PKV_BF16), 16-byte aligned.
 *   slot_mapping   device int64 [num_tokens]; negative = do not write.
 *   k_scale, v_scale device fp32 [num_kv_heads], > 0.
 *   k_cache, v_cache device uint8 pools as laid out above, 16-byte aligned.
 *   device_error   device int32 or NULL; PKV_DEVERR_SLOT for slots outside
 *                  [0, num_pages * page_size) (the token is skipped).
 * page_size is 16, 32, 64, 128 or 256.  num_tokens == 0 is a no-op.  Two
 * tokens with the same slot race.
 */
pkv_status pkv_kv_append_fp8(const void *k_new, const void *v_new, int in_dtype,
                             int64_t num_tokens, int num_kv_heads, int head_dim,
                             const int64_t *slot_mapping,
                             const float *k_scale, const float *v_scale,
                             uint8_t *k_cache, uint8_t *v_cache,
                             int64_t num_pages, int page_size,
                             int32_t *device_error, cudaStream_t stream);

/*
 * kv_calibrate -- on-device KV-scale calibration ([G] §3.2: every attention
 * layer keeps a running maximum of the KV values seen during prefill and
 * quantises new KV with the scale derived from it; [G] §3.1: scale =
 * absmax / 448 with a 1e-12 floor).
 *
 *   k_running_max[h] = max(k_running_max[h], |k_new[t][h][d]| over t, d)
 *   (same for V; NaN values are ignored), then, if k_scale/v_scale are given,
 *   k_scale[h] = max(k_running_max[h] / 448, 1e-12) (IEEE fp32 division).
 *
 *   k_new, v_new       device [num_tokens][num_kv_heads][head_dim], PKV_F32 or
 *                      PKV_BF16, 16-byte aligned.
 *   *_running_max      device fp32 [num_kv_heads], caller-owned state: zero it
 *                      when a layer starts calibrating; updated in place.
 *   k_scale, v_scale   device fp32 [num_kv_heads] outputs, or both NULL.
 * Calls on one stream compose: the maxima of several prefill batches equal
 * the maximum over their union.
 */
pkv_status pkv_kv_calibrate(const void *k_new, const void *v_new, int in_dtype,
                            int64_t num_tokens, int num_kv_heads, int head_dim,
                            float *k_running_max, float *v_running_max,
                            float *k_scale, float *v_scale, cudaStream_t stream);

/*
 * Workspace bytes pkv_paged_gqa_decode needs on the current device for a
 * call with these sizes whose seq_lens are all <= max_seq_len (partial
 * softmax states of the split-K pass: one slot per split-K worker plus one
 * per (sequence, kv head)).  Returns 0 for sizes the library rejects.
 * max_ctas as in pkv_paged_gqa_decode.  Independent of max_seq_len and of
 * the split weights (about 8 MB at batch 64, 8 kv heads, G = 8 on a 152-SM
 * GPU).
 */
size_t pkv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                 int head_dim, int max_seq_len, int page_size, int max_ctas);

/*
 * paged_gqa_decode -- one decode step of grouped-query attention over the
 * paged FP8 cache ([G] §1.2 GQA; [N] §2.2/§5.2 paging; [N] §3.2 the whole
 * cache is read every step).
 *
 * For every sequence b < batch and query head i < num_q_heads, with
 * G = num_q_heads / num_kv_heads, h = i / G and L = seq_lens[b]:
 *     s_t = sm_scale * sum_d q[b][i][d] * E4M3(k_cache[pg(t)][h][row(t)][d]) * k_scale[h]
 *     w_t = softmax_t(s_t)                              for t < L
 *     out[b][i][d] = sum_t w_t * E4M3(v_cache[pg(t)][h][row(t)][d]) * v_scale[h]
 * where, with P = page_size and P_b the sequence's page size (P unless
 * seq_page_sizes is given), pg(t) = block_table[b][t / P_b] + (t % P_b) / P
 * and row(t) = t % P: a page of P_b tokens is a run of P_b / P consecutive
 * pool pages, and its table entry is the first of them ([N] §3.2: 16-token
 * pages for short sequences, 64-token pages for long ones).  L == 0 gives a
 * zero row.  Long contexts are split across warps (split-K /
 * flash-decoding); no warp chains more than 128 chunks of 16 tokens on the
 * tensor cores (longer ranges fold their accumulator into their partial
 * state in fp32 every 128 chunks), and a second kernel merges the partial softmax
 * states exactly (log-sum-exp) in a fixed order: results are deterministic
 * run to run and independent of where the pages sit in the pool.  Two kernel
 * launches (the second is a programmatic dependent launch that overlaps the
 * first one's tail).
 *
 *   q              device bf16 [batch][num_q_heads][head_dim] (|q| < 65504).
 *   k_cache, v_cache device uint8 pools (layout above), 16-byte aligned.
 *   k_scale, v_scale device fp32 [num_kv_heads].
 *   block_table    device int32 [batch][max_pages_per_seq].
 *   seq_lens       device int32 [batch]; must satisfy
 *                  0 <= seq_lens[b] <= min(max_seq_len, max_pages_per_seq * P_b)
 *                  (violations set PKV_DEVERR_SEQLEN and are clamped).
 *   max_seq_len    host bound of seq_lens (lengths above it are clamped
 *                  and flagged); 0 means max_pages_per_seq * page_size
 *                  (pass the real bound when seq_page_sizes is given).
 *   seq_page_sizes device int32 [batch] or NULL: tokens per page of each
 *                  sequence, a power of two in [page_size, 256] (others set
 *                  PKV_DEVERR_PAGESIZE and the sequence reads as empty).
 *   head_dim       128.  page_size 16, 32, 64, 128 or 256.  G in 1..8.
 *   sm_scale       softmax scale, normally 1/sqrt(head_dim).
 *   out            device [batch][num_q_heads][head_dim], out_dtype
 *                  PKV_BF16 (bf16, RNE of the fp32 result) or PKV_F32.
 *   workspace      device, >= pkv_decode_workspace_size(batch, num_q_heads,
 *                  num_kv_heads, head_dim, max_seq_len, page_size, max_ctas)
 *                  bytes, 256-byte aligned: a header, per-(sequence, kv
 *                  head) records, then the partial states.  Contents need no
 *                  initialisation; one workspace must not be shared by calls
 *                  that overlap on the GPU.
 *   device_error   device int32 or NULL (bits above).
 *   max_ctas       0 = one persistent CTA per resident slot on the device;
 *                  > 0 caps the CTA count (changes the split, not the math).
 */
pkv_status pkv_paged_gqa_decode(const void *q,
                                const uint8_t *k_cache, const uint8_t *v_cache,
                                const float *k_scale, const float *v_scale,
                                const int32_t *block_table, int max_pages_per_seq,
                                const int32_t *seq_lens, int max_seq_len,
                                const int32_t *seq_page_sizes,
                                int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                int page_size, int64_t num_pages, float sm_scale,
                                void *out, int out_dtype,
                                void *workspace, size_t workspace_bytes,
                                int32_t *device_error, int max_ctas, cudaStream_t stream);

/*
 * append_decode_fp8 -- one whole decode step in one call: the kv_append_fp8
 * of the step's new tokens fused into paged_gqa_decode ([G] §3.2: new K/V are
 * quantised with the layer's scale as they are produced; [N] §3.2 decode).
 *
 * For every sequence b with L = seq_lens[b] (the length AFTER this step's
 * tokens) and j < n_new, token position t = L - n_new + j:
 *     k_cache[pg(t)][h][row(t)][d] = E4M3(k_new[b][j][h][d] / k_scale[h])
 * (same for V, same rounding as pkv_kv_append_fp8; pg and row as in
 * pkv_paged_gqa_decode), then exactly the attention of pkv_paged_gqa_decode
 * over t < L.  Page bytes and outputs are bit-identical to calling
 * pkv_kv_append_fp8 with slot = block_table[b][t / P_b] * P + t % P_b
 * followed by pkv_paged_gqa_decode.  Each new token is written by the warp
 * that later reads its page, so no extra launch or grid-wide ordering is
 * needed.
 *
 *   k_new, v_new   device [batch][n_new][num_kv_heads][head_dim], in_dtype
 *                  PKV_F32 or PKV_BF16, 16-byte aligned (unused if n_new == 0).
 *   n_new          tokens appended per sequence (>= 0); seq_lens[b] < n_new
 *                  drops the missing positions and sets PKV_DEVERR_SEQLEN.
 *   The pages receiving new tokens must not be shared with another sequence
 *   of the same call (prefix-shared pages are read-only).
 *   Everything else as in pkv_paged_gqa_decode (the caches are written).
 */
pkv_status pkv_append_decode_fp8(const void *k_new, const void *v_new, int in_dtype, int n_new,
                                 const void *q, uint8_t *k_cache, uint8_t *v_cache,
                                 const float *k_scale, const float *v_scale,
                                 const int32_t *block_table, int max_pages_per_seq,
                                 const int32_t *seq_lens, int max_seq_len,
                                 const int32_t *seq_page_sizes,
                                 int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                 int page_size, int64_t num_pages, float sm_scale,
                                 void *out, int out_dtype,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t *device_error, int max_ctas, cudaStream_t stream);

/*
 * Split weights -- how the decode call shares the cache among its workers.
 * Decode is bound by the rate at which the whole cache streams in ([N] §3.2),
 * so the call ends when its slowest worker does.  The workers are the warps
 * of a persistent grid; by default every warp takes an equal share of the
 * list of 16-token chunks.  The SMs of one GPU do not all stream equally
 * fast, and the grid's CTAs land on the same SMs call after call, so equal
 * shares leave the fast SMs idle while the slow ones finish.  With weights,
 * CTA c's four warps take shares proportional to weights[c]: with
 * C(w) = 4 * (weights[0] + ... + weights[c-1]) + j * weights[c] for warp j
 * of CTA c, worker w covers list positions [T * C(w) / CT, T * C(w + 1) / CT)
 * of the T chunks, CT = C(4n).  Equal weights give exactly the default split.
 * (The list the split cuts counts 3 empty chunks after every sequence's
 * chunks of a kv head, the cost of the extra piece a range holding a
 * sequence's end carries; a range's real edges are where its edges in that
 * list fall.  Only when every range then holds a chunk: T * min weight >= CT.)
 * The math is unchanged; the pieces the split cuts (and so the last bits of
 * the result, within the accuracy bound) depend on the weights, and stay
 * deterministic for fixed weights.
 *
 * Weights belong to the device's current context: after a cudaDeviceReset
 * they no longer apply (the calls split evenly and
 * pkv_decode_get_split_weights reports none) until they are installed again.
 * (A process that resets a device should restart before decoding on it
 * again: the split-K merge kernel's raised shared-memory limit is not set up
 * anew, so decode calls with more than 6 query heads per kv head then fail
 * with PKV_ERR_CUDA.  Everything else is set up again on the next call.)
 *
 * pkv_decode_set_split_weights installs n weights, each an integer in
 * [768, 1280] (1024 +- 25%), for the current device; they apply to decode calls
 * (pkv_paged_gqa_decode, pkv_append_decode_fp8 and the allocation-free entry
 * point) whose grid has exactly n CTAs, and the others split evenly.  n == 0
 * removes them.  Copies n + 1 integers to device memory the decode kernels
 * read, synchronously: do not call it while a decode call is in flight on
 * the device, or during stream capture.  Errors: PKV_ERR_SHAPE (n outside
 * [0, 1024] or a weight outside [768, 1280]), PKV_ERR_NULL, PKV_ERR_CUDA.
 *
 * pkv_decode_get_split_weights copies the current device's weights to
 * weights[0 .. *n) (*n = 0: none; PKV_ERR_SHAPE if *n > capacity).
 *
 * pkv_decode_calibrate_split measures them: it runs `rounds` (1..64) times
 * four decode calls with the given arguments (as pkv_paged_gqa_decode; out
 * and workspace are written, max_ctas sets the grid), each timed per CTA
 * with the global timer, synchronising `stream` after each; every round
 * sets each CTA's weight to the share it streams in the time all CTAs take
 * together, and the result is the average of the rounds after the first
 * (the first moves the weights from equal to near the balance).  Starts
 * from equal weights, leaves the result installed (and
 * copies it to weights_out[0 .. n), if weights_out is given, with n in
 * *n_out).  On an error the device's weights are removed.  A setup-time
 * call: a few ms of GPU time plus host synchronisation; not capturable.
 */
pkv_status pkv_decode_set_split_weights(const uint16_t *weights, int n);
/*
 * The CUDA runtime error (cudaError_t value) behind the calling thread's last
 * PKV_ERR_CUDA status, 0 if none; with name given, *name points to a text
 * naming the error and the call that failed (owned by the library, valid
 * until the thread's next pkv_last_cuda_error call).
 */
int pkv_last_cuda_error(const char **name);
pkv_status pkv_decode_get_split_weights(uint16_t *weights, int capacity, int *n);
pkv_status pkv_decode_calibrate_split(const void *q,
                                      const uint8_t *k_cache, const uint8_t *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_table, int max_pages_per_seq,
                                      const int32_t *seq_lens, int max_seq_len,
                                      const int32_t *seq_page_sizes,
                                      int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                      int page_size, int64_t num_pages, float sm_scale,
                                      void *out, int out_dtype,
                                      void *workspace, size_t workspace_bytes, int max_ctas,
                                      int rounds, uint16_t *weights_out, int capacity, int *n_out,
                                      cudaStream_t stream);

/*
 * paged_gqa_decode without a caller workspace, for callers that cannot
 * allocate device memory (a serving engine that owns every byte of device
 * memory through its own pool, a plugin that must not bypass its host
 * runtime's allocator, a latency-critical loop that cannot pay for an
 * allocation).  No counterpart on the pages: it is an interface variant, the
 * computation is exactly pkv_paged_gqa_decode's.
 *
 * Same arguments and results as pkv_paged_gqa_decode minus the workspace.
 * The split-K scratch lives in a fixed array inside the library image,
 * pkv_decode_noalloc_scratch_bytes() bytes (16 MiB).  Under CUDA's default
 * lazy module loading a GPU holds the array from the first call on it (the
 * first launch of any of this library's kernels there) until the process
 * exits; with eager loading, from library load.  The call allocates nothing.
 * It accepts exactly the sizes for which pkv_decode_workspace_size(...) with
 * the same arguments is at most pkv_decode_noalloc_scratch_bytes(), and
 * returns PKV_ERR_WORKSPACE for larger ones; that bound depends on the GPU in
 * use (its SM count sets the number of split-K workers), so query it rather
 * than assume a batch limit.
 * All calls share the array: calls that overlap on the GPU (two streams, or
 * unordered host threads) race and corrupt each other's results; calls
 * ordered on one stream are safe.  The array keeps the previous call's
 * contents, which the decode never reads before writing.  The first call on
 * each device looks up the array's device address (with that device current)
 * and caches it: make that first call before any stream capture.  After
 * cudaDeviceReset the next call looks the address up again.
 */
pkv_status pkv_paged_gqa_decode_noalloc(const void *q,
                                        const uint8_t *k_cache, const uint8_t *v_cache,
                                        const float *k_scale, const float *v_scale,
                                        const int32_t *block_table, int max_pages_per_seq,
                                        const int32_t *seq_lens, int max_seq_len,
                                        const int32_t *seq_page_sizes,
                                        int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                        int page_size, int64_t num_pages, float sm_scale,
                                        void *out, int out_dtype,
                                        int32_t *device_error, int max_ctas, cudaStream_t stream);

/* Size in bytes of the fixed scratch array pkv_paged_gqa_decode_noalloc uses. */
size_t pkv_decode_noalloc_scratch_bytes(void);

/*
 * paged_prefill -- chunked-prefill attention over the paged FP8 cache ([N]
 * §2.2: a long prompt is prefilled in chunks, 8 x 16K for a 128K prompt, and
 * each chunk's KV joins the cache; [G] §1.2 GQA).  Call it after
 * pkv_kv_append_fp8 has written the chunk's own K/V into the pages.
 *
 * Sequence b owns query rows cu_q[b] .. cu_q[b+1] - 1 (n_b rows) of q; with
 * L = seq_lens[b] (the length INCLUDING the chunk), row c sits at position
 * p = L - n_b + c, and for every query head i (h = i / G, G = num_q_heads /
 * num_kv_heads):
 *     s_t = sm_scale * sum_d q[cu_q[b]+c][i][d] * E4M3(k_cache[pg(t)][h][row(t)][d]) * k_scale[h]
 *     w_t = softmax_t(s_t)                              for t <= p (causal)
 *     out[cu_q[b]+c][i][d] = sum_t w_t * E4M3(v_cache[pg(t)][h][row(t)][d]) * v_scale[h]
 * with pg and row as in pkv_paged_gqa_decode (per-sequence page sizes
 * included).  A chunk of one query is exactly one decode step.  Two
 * launches: the visible K/V of every sequence with a non-empty chunk are
 * first widened once from the pages to 16 bits (exact: K as bf16, V as f16)
 * into the workspace, packed sequence after sequence, then the attention
 * runs on the tcgen05 tensor cores (q K^T on bf16 operands; the softmax
 * weights as two f16 parts against f16 V; fp32 accumulation, the PV
 * accumulator added into a second fp32 accumulator every 32 key tiles).
 * Deterministic.
 *
 *   q              device bf16 [total_q][num_q_heads][head_dim], 16-byte
 *                  aligned.
 *   cu_q           device int32 [batch + 1], non-decreasing, cu_q[0] = 0,
 *                  cu_q[batch] <= total_q.
 *   total_q        rows of q and out.
 *   max_q_len      an upper bound of the chunk lengths n_b (sizes the grid).
 *   max_kv_len     an upper bound of seq_lens.
 *   max_total_kv   0, or an upper bound of the sum of seq_lens[b] over the
 *                  sequences with a non-empty chunk (with max_kv_len, sizes
 *                  the workspace: a batch of one long prompt and many short
 *                  chunks needs room for the long one only once).
 *   seq_lens       device int32 [batch]; a sequence with n_b > max_q_len,
 *                  seq_lens[b] < n_b, seq_lens[b] > max_kv_len or beyond
 *                  its table row, or inconsistent cu_q, sets
 *                  PKV_DEVERR_SEQLEN and its rows are not written; so does a
 *                  sequence whose widened copy would not fit the workspace
 *                  (the sum bound exceeded).
 *   seq_page_sizes device int32 [batch] or NULL, as in pkv_paged_gqa_decode
 *                  (an invalid entry sets PKV_DEVERR_PAGESIZE and the
 *                  sequence's rows are not written).
 *   block_table    entries of pages the chunk's positions need must lie in
 *                  [0, num_pages); others set PKV_DEVERR_PAGE and the page
 *                  reads as zeros.
 *   out            device [total_q][num_q_heads][head_dim], PKV_BF16 or
 *                  PKV_F32, 16-byte aligned.  Rows outside every chunk are
 *                  not written.
 *   workspace      device, >= pkv_prefill_workspace_size(batch, num_kv_heads,
 *                  max_kv_len, max_total_kv) bytes, 256-byte aligned: the
 *                  sequences' region offsets, then the 16-bit copies of K
 *                  and V (overwritten every call; must not be shared by calls
 *                  that overlap on the GPU).
 *   sm_scale       softmax scale, > 0 (normally 1/sqrt(head_dim)); k_scale
 *                  entries must be positive (calibration gives absmax/448,
 *                  floored at 1e-12).
 *   Caches, scales, head_dim (128), page sizes, G (1..8) and device_error as
 *   in pkv_paged_gqa_decode.  batch * num_kv_heads * ceil(max_q_len /
 *   (128 / G)) must be below 2^31, and so must the copies' rows.
 */
size_t pkv_prefill_workspace_size(int batch, int num_kv_heads, int max_kv_len, int64_t max_total_kv);

pkv_status pkv_paged_prefill(const void *q, const int32_t *cu_q, int total_q, int max_q_len,
                             const uint8_t *k_cache, const uint8_t *v_cache,
                             const float *k_scale, const float *v_scale,
                             const int32_t *block_table, int max_pages_per_seq,
                             const int32_t *seq_lens, const int32_t *seq_page_sizes,
                             int batch, int max_kv_len, int64_t max_total_kv,
                             int num_q_heads, int num_kv_heads, int head_dim,
                             int page_size, int64_t num_pages, float sm_scale,
                             void *out, int out_dtype,
                             void *workspace, size_t workspace_bytes,
                             int32_t *device_error, cudaStream_t stream);

/*
 * read_device_error -- read (and optionally clear) a device error word after
 * the work already enqueued on `stream`.
 *
 *   device_error   device int32, the word passed to the calls above.
 *   clear          non-zero: reset the word to 0 after reading it (enqueued
 *                  on `stream`, so it is ordered before later work there).
 *   code           host int32 out: the word's bits (PKV_DEVERR_*).
 * Unlike every other call this one synchronises `stream` (it waits for the
 * word).  Returns PKV_ERR_NULL / PKV_ERR_ALIGN for bad pointers and
 * PKV_ERR_CUDA if the copy or the wait fails (for example after a sticky
 * CUDA error of an earlier launch).
 */
pkv_status pkv_read_device_error(const int32_t *device_error, int clear, int32_t *code,
                                 cudaStream_t stream);

/*
 * Test facility for the failure-detection tests, not for production use.
 * After pkv_test_withhold_load(w) with w >= 0, decode worker warp w never
 * loads its first page, and in pkv_paged_prefill the CTA of grid block w
 * never loads its first K tile: a pipeline wait runs out after about 2 s and
 * the call sets PKV_DEVERR_TIMEOUT (outputs undefined), without faulting or
 * hanging the GPU.  w < 0 (the state at load) turns it off.  Process-wide;
 * applies to calls made after it returns.
 */
void pkv_test_withhold_load(int index);

/* Human-readable name of a status code (static string). */
const char *pkv_status_string(pkv_status status);

/* Library ABI version: (major << 16) | minor. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDFP8_H */
