// C entry points: argument checks on the host, TMA tensor descriptions of the
// page pools, grid sizing and launches.  Nothing here allocates device memory.
#include <math.h>
#include <stdio.h>

#include <atomic>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "context.h"
#include "internal.h"

namespace pkv {

namespace {

std::mutex g_mu;
std::map<int, int> g_sm_count;                              // device -> SMs
std::map<std::tuple<int, const void *, size_t>, int> g_occupancy;   // (device, kernel, smem) -> CTAs per SM
// (context, kernel) -> the kernel's dynamic shared memory limit set so far
// in that context (only ever raised: every page size runs the same kernel, so
// a limit per page size would let one page size's smaller setting undercut
// another's launch; a device reset starts a new context at the default).
std::map<std::tuple<unsigned long long, const void *>, size_t> g_smem_attr;
std::atomic<int> g_withhold{-1};                            // failure-detection test facility (-1 = off)

// Weighted split of each device: the per-CTA weights for one grid size (the
// prefix sums live in the decode module's device table).  Absent: even split.
struct SplitState {
    std::vector<uint16_t> weights;
    long long ct = 0;                                       // 4 * sum of the weights
    int wmin = 0, wmax = 0;
    unsigned long long ctx = 0;                             // context the device table was written in (0: unknown)
};
std::map<int, SplitState> g_split;                          // device -> weights

// The device's installed weights, or nullptr.  Weights uploaded in an earlier
// context of the device (before a device reset) are gone from the device
// table the kernels read, so they are dropped: the device splits evenly until
// weights are installed again.  Call with g_mu held.
const SplitState *live_split(int dev)
{
    auto it = g_split.find(dev);
    if (it == g_split.end())
        return nullptr;
    unsigned long long ctx = 0;
    if (it->second.ctx != 0 && current_context_id(&ctx) && ctx != it->second.ctx) {
        g_split.erase(it);
        return nullptr;
    }
    return &it->second;
}
thread_local int t_last_cuda = 0;                           // error behind this thread's last PKV_ERR_CUDA
thread_local const char *t_last_site = "";                  // the call that failed
thread_local char t_last_text[160];

pkv_status cuda_failed(cudaError_t e, const char *site = "")
{
    t_last_cuda = e == cudaSuccess ? static_cast<int>(cudaErrorUnknown) : static_cast<int>(e);
    t_last_site = site;
    return PKV_ERR_CUDA;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

// A pool [num_pages][hkv][P][128] bytes seen as a 3-D tensor (128 bytes, P rows,
// num_pages*hkv tiles); one box = 16 rows (one chunk) of one page of one kv
// head, 128-byte swizzled.
bool make_page_map(CUtensorMap *tm, const uint8_t *pool, int64_t num_pages, int hkv, int P)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(P),
                                static_cast<cuuint64_t>(num_pages) * static_cast<cuuint64_t>(hkv)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(P) * kHeadDim};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), 16u, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Queries [total_q][hq][128] bf16 as a 3-D tensor (128 dims, hq heads, total_q
// rows); one box = 64 dims of the G heads of one kv head for tpt rows, 128-byte
// swizzled, which is the layout the tensor cores read as a K-major operand.
bool make_q_map(CUtensorMap *tm, const void *q, int total_q, int hq, int group, int tpt)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(hq),
                                static_cast<cuuint64_t>(total_q)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                                   static_cast<cuuint64_t>(hq) * kHeadDim * 2};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tpt)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The 16-bit copies of K (bf16) or V (f16), [rows][128], as a 3-D tensor
// (128 dims, rows keys, 1); one box = 64 dims of 128 keys, 128-byte swizzled:
// one column block of an MMA operand tile.
bool make_kv16_map(CUtensorMap *tm, const void *base, long long rows, CUtensorMapDataType dtype)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows), 1};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                                   static_cast<cuuint64_t>(rows) * kHeadDim * 2};
    const cuuint32_t box[3] = {64u, 128u, 1u};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return -1;
    return dev;
}

}  // namespace

int device_sm_count()
{
    const int dev = current_device();
    if (dev < 0)
        return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_sm_count.find(dev);
    if (it != g_sm_count.end())
        return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    g_sm_count[dev] = n;
    return n;
}

// Persistent grid: every resident CTA slot on the device (capped by max_ctas).
int decode_num_ctas(int page_size, int batch, int max_ctas)
{
    const int dev = current_device();
    const int sms = device_sm_count();
    if (dev < 0 || sms <= 0) {
        cuda_failed(cudaGetLastError(), "device query");
        return 0;
    }
    const size_t smem = decode_smem_bytes(page_size, batch);
    const void *kern = decode_kernel_for(page_size);
    int per_sm = 0;
    {
        unsigned long long ctx = 0;
        const bool known = current_context_id(&ctx);   // (no id yet: set the limit, remember nothing)
        std::lock_guard<std::mutex> lk(g_mu);
        auto key_attr = std::make_tuple(ctx, kern);
        auto ia = known ? g_smem_attr.find(key_attr) : g_smem_attr.end();
        if (ia == g_smem_attr.end() || ia->second < smem) {
            const cudaError_t e =
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) {
                cuda_failed(e, "cudaFuncSetAttribute (decode shared memory)");
                return 0;
            }
            if (known)
                g_smem_attr[key_attr] = smem;
        }
        auto key = std::make_tuple(dev, kern, smem);
        auto it = g_occupancy.find(key);
        if (it != g_occupancy.end()) {
            per_sm = it->second;
        } else {
            const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
            if (e != cudaSuccess) {
                cuda_failed(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor (decode)");
                return 0;
            }
            g_occupancy[key] = per_sm;
        }
    }
    if (per_sm <= 0) {
        cuda_failed(cudaErrorInvalidConfiguration, "decode occupancy is 0 CTAs per SM");
        return 0;
    }
    int c = per_sm * sms;
    if (max_ctas > 0 && max_ctas < c)
        c = max_ctas;
    return c;
}

// Workspace: header and segment records, then one partial slot per worker
// plus one per segment (a piece is a worker's range within one segment; its
// slot is worker + the segment's rank in list order, distinct for every piece).  Independent of the
// sequence lengths.
size_t decode_workspace_bytes(int batch, int hq, int hkv, long long /*max_len*/, int num_ctas)
{
    const long long workers = static_cast<long long>(num_ctas) * kWarps;
    const size_t slots = static_cast<size_t>(workers) + static_cast<size_t>(batch) * hkv;
    const size_t bytes = slots * static_cast<size_t>(hq / hkv) * kPartialStride * sizeof(float);
    return decode_segment_bytes(batch, hkv) + ((bytes + 255) & ~size_t(255));
}

}  // namespace pkv

using namespace pkv;

namespace {

pkv_status check_decode_shape(int batch, int hq, int hkv, int head_dim, int page_size, int max_pages,
                              int64_t num_pages)
{
    if (batch < 0 || hq <= 0 || hkv <= 0 || max_pages <= 0 || num_pages <= 0)
        return PKV_ERR_SHAPE;
    if (hq % hkv != 0)
        return PKV_ERR_SHAPE;
    if (head_dim != kHeadDim || !page_size_ok(page_size))
        return PKV_ERR_UNSUPPORTED;
    if (hq / hkv > PKV_MAX_GROUP || batch > PKV_MAX_BATCH)
        return PKV_ERR_UNSUPPORTED;
    if (num_pages * static_cast<int64_t>(hkv) >= (int64_t(1) << 31) - 1)
        return PKV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_pages) * page_size >= (int64_t(1) << 31))
        return PKV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(batch) * max_pages >= (int64_t(1) << 40))
        return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// Effective bound of seq_lens: max_seq_len, or the table's capacity at the
// pool page size when max_seq_len is 0.
long long effective_max_len(int max_seq_len, int max_pages, int page_size)
{
    return max_seq_len > 0 ? max_seq_len : static_cast<long long>(max_pages) * page_size;
}

pkv_status decode_impl(const void *k_new, const void *v_new, int in_dtype, int n_new, const void *q, uint8_t *k_cache,
                       uint8_t *v_cache, const float *k_scale, const float *v_scale, const int32_t *block_table,
                       int max_pages_per_seq, const int32_t *seq_lens, int max_seq_len, const int32_t *seq_page_sizes,
                       int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
                       float sm_scale, void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                       int32_t *device_error, int max_ctas, cudaStream_t stream, bool probe = false,
                       int *probe_ctas = nullptr)
{
    pkv_status st = check_decode_shape(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_seq,
                                       num_pages);
    if (st != PKV_OK)
        return st;
    if (max_seq_len < 0)
        return PKV_ERR_SHAPE;
    if (seq_page_sizes && static_cast<int64_t>(max_pages_per_seq) * 256 >= (int64_t(1) << 31))
        return PKV_ERR_UNSUPPORTED;
    if (out_dtype != PKV_F32 && out_dtype != PKV_BF16)
        return PKV_ERR_DTYPE;
    if (!(sm_scale == sm_scale) || isinf(sm_scale))
        return PKV_ERR_SHAPE;
    if (batch == 0)
        return PKV_OK;
    if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !block_table || !seq_lens || !out)
        return PKV_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4) ||
        !aligned(device_error, 4) || !aligned(seq_page_sizes, 4))
        return PKV_ERR_ALIGN;
    if (!workspace || !aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;

    const long long max_len = effective_max_len(max_seq_len, max_pages_per_seq, page_size);
    if (max_len >= (int64_t(1) << 31))
        return PKV_ERR_UNSUPPORTED;
    const int ctas = decode_num_ctas(page_size, batch, max_ctas);
    if (ctas <= 0)
        return PKV_ERR_CUDA;                     // decode_num_ctas recorded the failing call
    if (workspace_bytes < decode_workspace_bytes(batch, num_q_heads, num_kv_heads, max_len, ctas))
        return PKV_ERR_WORKSPACE;

    alignas(64) CUtensorMap tm_k;
    alignas(64) CUtensorMap tm_v;
    if (!make_page_map(&tm_k, k_cache, num_pages, num_kv_heads, page_size) ||
        !make_page_map(&tm_v, v_cache, num_pages, num_kv_heads, page_size))
        return cuda_failed(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (page pools)");

    DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_table = block_table;
    a.max_pages = max_pages_per_seq;
    a.seq_lens = seq_lens;
    a.max_len = static_cast<int>(max_len);
    a.page_sizes = seq_page_sizes;
    a.batch = batch;
    a.hq = num_q_heads;
    a.hkv = num_kv_heads;
    a.group = num_q_heads / num_kv_heads;
    a.page_size = page_size;
    a.pool_log2 = 31 - __builtin_clz(static_cast<unsigned>(page_size));
    a.num_pages = num_pages;
    a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
    a.out = out;
    a.out_f32 = out_dtype == PKV_F32;
    a.k_new = k_new;
    a.v_new = v_new;
    a.new_bf16 = in_dtype == PKV_BF16;
    a.n_new = n_new;
    a.k_pool = k_cache;
    a.v_pool = v_cache;
    a.header = static_cast<DecodeHeader *>(workspace);
    a.segs = reinterpret_cast<SegRecord *>(static_cast<uint8_t *>(workspace) + sizeof(DecodeHeader));
    a.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + decode_segment_bytes(batch, num_kv_heads));
    a.err = device_error;
    a.num_ctas = ctas;
    // Test facility for the timeout path (pkv_test_withhold_load): that worker
    // warp skips its first page's loads, so its first wait runs out (about
    // 2 s) and the call reports PKV_DEVERR_TIMEOUT.  -1: no effect.
    a.withhold_worker = g_withhold.load(std::memory_order_relaxed);
    a.split = 0;
    a.split_ct = 0;
    a.split_wmin = a.split_wmax = 1;
    a.probe = probe ? 1 : 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const SplitState *live = live_split(current_device());
        if (live != nullptr && static_cast<int>(live->weights.size()) == ctas) {
            a.split = 1;
            a.split_ct = live->ct;
            a.split_wmin = live->wmin;
            a.split_wmax = live->wmax;
        }
    }
    if (probe_ctas)
        *probe_ctas = ctas;
    const size_t slot_bytes = static_cast<size_t>(a.group) * kPartialStride * sizeof(float);
    a.num_slots = static_cast<long long>((workspace_bytes - decode_segment_bytes(batch, num_kv_heads)) / slot_bytes);
    const char *site = "";
    const cudaError_t e = launch_paged_decode(a, tm_k, tm_v, page_size, stream, &site);
    return e == cudaSuccess ? PKV_OK : cuda_failed(e, site);
}

// Installs weights (n of them, each in [kSplitWeightMin, kSplitWeightMax]) for
// the current device; n == 0 removes them (even split).
pkv_status set_split(const uint16_t *weights, int n)
{
    if (n < 0 || n > kMaxSplitCtas || (n > 0 && !weights))
        return n < 0 || n > kMaxSplitCtas ? PKV_ERR_SHAPE : PKV_ERR_NULL;
    SplitState st;
    std::vector<uint32_t> prefix(static_cast<size_t>(n) + 1, 0u);
    st.wmin = kSplitWeightMax;
    st.wmax = kSplitWeightMin;
    for (int c = 0; c < n; ++c) {
        const int w = weights[c];
        if (w < kSplitWeightMin || w > kSplitWeightMax)
            return PKV_ERR_SHAPE;
        prefix[c + 1] = prefix[c] + static_cast<uint32_t>(w);
        st.wmin = w < st.wmin ? w : st.wmin;
        st.wmax = w > st.wmax ? w : st.wmax;
    }
    const int dev = current_device();
    if (dev < 0)
        return cuda_failed(cudaGetLastError());
    std::lock_guard<std::mutex> lk(g_mu);
    if (n == 0) {
        g_split.erase(dev);
        return PKV_OK;
    }
    const cudaError_t e = upload_split_prefix(prefix.data(), n);
    if (e != cudaSuccess)
        return cuda_failed(e);
    unsigned long long ctx = 0;
    st.ctx = current_context_id(&ctx) ? ctx : 0;
    st.weights.assign(weights, weights + n);
    st.ct = static_cast<long long>(kWarps) * prefix[n];
    g_split[dev] = st;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_version(void)
{
    return (1 << 16) | 0;
}

void pkv_test_withhold_load(int index)
{
    g_withhold.store(index < 0 ? -1 : index, std::memory_order_relaxed);
}

pkv_status pkv_read_device_error(const int32_t *device_error, int clear, int32_t *code, cudaStream_t stream)
{
    if (!device_error || !code)
        return PKV_ERR_NULL;
    if (!aligned(device_error, 4))
        return PKV_ERR_ALIGN;
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, device_error, sizeof(word), cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess)
        return cuda_failed(e);
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return cuda_failed(e);
    *code = word;
    if (clear) {
        e = cudaMemsetAsync(const_cast<int32_t *>(device_error), 0, sizeof(word), stream);
        if (e != cudaSuccess)
            return cuda_failed(e);
    }
    return PKV_OK;
}

const char *pkv_status_string(pkv_status s)
{
    switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_SHAPE: return "invalid or inconsistent sizes";
    case PKV_ERR_DTYPE: return "unknown dtype code";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration (head_dim, page size, group, batch or pool size)";
    case PKV_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case PKV_ERR_CUDA: return "CUDA call or kernel launch failed";
    case PKV_ERR_ALIGN: return "pointer not aligned as required";
    default: return "unknown status";
    }
}

pkv_status pkv_kv_append_fp8(const void *k_new, const void *v_new, int in_dtype, int64_t num_tokens,
                             int num_kv_heads, int head_dim, const int64_t *slot_mapping, const float *k_scale,
                             const float *v_scale, uint8_t *k_cache, uint8_t *v_cache, int64_t num_pages,
                             int page_size, int32_t *device_error, cudaStream_t stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || num_pages <= 0)
        return PKV_ERR_SHAPE;
    if (in_dtype != PKV_F32 && in_dtype != PKV_BF16)
        return PKV_ERR_DTYPE;
    if (head_dim != kHeadDim || !page_size_ok(page_size))
        return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0)
        return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_scale || !v_scale || !k_cache || !v_cache)
        return PKV_ERR_NULL;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8) || !aligned(k_scale, 4) || !aligned(v_scale, 4) ||
        !aligned(device_error, 4))
        return PKV_ERR_ALIGN;
    AppendArgs a;
    a.k_new = k_new;
    a.v_new = v_new;
    a.in_bf16 = in_dtype == PKV_BF16;
    a.num_tokens = num_tokens;
    a.hkv = num_kv_heads;
    a.slots = slot_mapping;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_pages = num_pages;
    a.page_size = page_size;
    a.err = device_error;
    const cudaError_t e = launch_kv_append(a, stream);
    return e == cudaSuccess ? PKV_OK : cuda_failed(e);
}

size_t pkv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim, int max_seq_len,
                                 int page_size, int max_ctas)
{
    if (check_decode_shape(batch, num_q_heads, num_kv_heads, head_dim, page_size, 1, 1) != PKV_OK ||
        max_seq_len < 0)
        return 0;
    const int ctas = decode_num_ctas(page_size, batch, max_ctas);
    if (ctas <= 0)
        return 0;
    return decode_workspace_bytes(batch, num_q_heads, num_kv_heads, max_seq_len, ctas);
}

pkv_status pkv_paged_gqa_decode(const void *q, const uint8_t *k_cache, const uint8_t *v_cache, const float *k_scale,
                                const float *v_scale, const int32_t *block_table, int max_pages_per_seq,
                                const int32_t *seq_lens, int max_seq_len, const int32_t *seq_page_sizes, int batch,
                                int num_q_heads, int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
                                float sm_scale, void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                                int32_t *device_error, int max_ctas, cudaStream_t stream)
{
    return decode_impl(nullptr, nullptr, PKV_F32, 0, q, const_cast<uint8_t *>(k_cache), const_cast<uint8_t *>(v_cache),
                       k_scale, v_scale, block_table, max_pages_per_seq, seq_lens, max_seq_len, seq_page_sizes, batch,
                       num_q_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale, out, out_dtype, workspace,
                       workspace_bytes, device_error, max_ctas, stream);
}

pkv_status pkv_append_decode_fp8(const void *k_new, const void *v_new, int in_dtype, int n_new, const void *q,
                                 uint8_t *k_cache, uint8_t *v_cache, const float *k_scale, const float *v_scale,
                                 const int32_t *block_table, int max_pages_per_seq, const int32_t *seq_lens,
                                 int max_seq_len, const int32_t *seq_page_sizes, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, int page_size, int64_t num_pages, float sm_scale,
                                 void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                                 int32_t *device_error, int max_ctas, cudaStream_t stream)
{
    if (n_new < 0)
        return PKV_ERR_SHAPE;
    if (in_dtype != PKV_F32 && in_dtype != PKV_BF16)
        return PKV_ERR_DTYPE;
    if (n_new > 0 && batch > 0) {
        if (!k_new || !v_new)
            return PKV_ERR_NULL;
        if (!aligned(k_new, 16) || !aligned(v_new, 16))
            return PKV_ERR_ALIGN;
    }
    return decode_impl(n_new > 0 ? k_new : nullptr, n_new > 0 ? v_new : nullptr, in_dtype, n_new, q, k_cache, v_cache,
                       k_scale, v_scale, block_table, max_pages_per_seq, seq_lens, max_seq_len, seq_page_sizes, batch,
                       num_q_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale, out, out_dtype, workspace,
                       workspace_bytes, device_error, max_ctas, stream);
}

pkv_status pkv_decode_set_split_weights(const uint16_t *weights, int n)
{
    return set_split(weights, n);
}

int pkv_last_cuda_error(const char **name)
{
    if (name) {
        snprintf(t_last_text, sizeof(t_last_text), "%s%s%s",
                 t_last_cuda ? cudaGetErrorName(static_cast<cudaError_t>(t_last_cuda)) : "cudaSuccess",
                 *t_last_site ? " in " : "", t_last_site);
        *name = t_last_text;
    }
    return t_last_cuda;
}

pkv_status pkv_decode_get_split_weights(uint16_t *weights, int capacity, int *n)
{
    if (!n || capacity < 0 || (capacity > 0 && !weights))
        return PKV_ERR_NULL;
    const int dev = current_device();
    if (dev < 0)
        return cuda_failed(cudaGetLastError());
    std::lock_guard<std::mutex> lk(g_mu);
    const SplitState *live = live_split(dev);
    const int have = live == nullptr ? 0 : static_cast<int>(live->weights.size());
    *n = have;
    if (have > capacity)
        return PKV_ERR_SHAPE;
    for (int c = 0; c < have; ++c)
        weights[c] = live->weights[c];
    return PKV_OK;
}

pkv_status pkv_decode_calibrate_split(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                      const float *k_scale, const float *v_scale, const int32_t *block_table,
                                      int max_pages_per_seq, const int32_t *seq_lens, int max_seq_len,
                                      const int32_t *seq_page_sizes, int batch, int num_q_heads, int num_kv_heads,
                                      int head_dim, int page_size, int64_t num_pages, float sm_scale, void *out,
                                      int out_dtype, void *workspace, size_t workspace_bytes, int max_ctas,
                                      int rounds, uint16_t *weights_out, int capacity, int *n_out,
                                      cudaStream_t stream)
{
    if (rounds < 1 || rounds > 64)
        return PKV_ERR_SHAPE;
    if (batch <= 0)
        return PKV_ERR_SHAPE;
    if (check_decode_shape(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_seq, num_pages) !=
        PKV_OK)
        return PKV_ERR_SHAPE;
    const int ctas = decode_num_ctas(page_size, batch, max_ctas);
    if (ctas <= 0)
        return PKV_ERR_CUDA;
    if (ctas > kMaxSplitCtas)
        return PKV_ERR_UNSUPPORTED;
    constexpr int kCallsPerRound = 4;
    constexpr double kMean = 0.5 * (kSplitWeightMin + kSplitWeightMax);
    auto quantise = [](double v) {
        v = v < kSplitWeightMin ? kSplitWeightMin : (v > kSplitWeightMax ? kSplitWeightMax : v);
        return static_cast<uint16_t>(v + 0.5);
    };
    std::vector<double> wd(static_cast<size_t>(ctas), kMean), avg(static_cast<size_t>(ctas), 0.0);
    std::vector<uint16_t> w(static_cast<size_t>(ctas), quantise(kMean));
    std::vector<unsigned long long> times(static_cast<size_t>(ctas) * 2);
    int n_avg = 0;
    pkv_status st = set_split(w.data(), ctas);
    for (int r = 0; r < rounds && st == PKV_OK; ++r) {
        // Finish (F) and start (S) of every CTA, relative to the first CTA's start.
        std::vector<double> F(static_cast<size_t>(ctas), 0.0), S(static_cast<size_t>(ctas), 0.0);
        for (int call = 0; call < kCallsPerRound && st == PKV_OK; ++call) {
            int used = 0;
            const cudaError_t ce = clear_split_probe(ctas, stream);
            if (ce != cudaSuccess) {
                st = cuda_failed(ce);
                break;
            }
            st = decode_impl(nullptr, nullptr, PKV_F32, 0, q, const_cast<uint8_t *>(k_cache),
                             const_cast<uint8_t *>(v_cache), k_scale, v_scale, block_table, max_pages_per_seq,
                             seq_lens, max_seq_len, seq_page_sizes, batch, num_q_heads, num_kv_heads, head_dim,
                             page_size, num_pages, sm_scale, out, out_dtype, workspace, workspace_bytes, nullptr,
                             max_ctas, stream, true, &used);
            if (st != PKV_OK)
                break;
            cudaError_t re = used != ctas ? cudaErrorInvalidValue : cudaStreamSynchronize(stream);
            if (re == cudaSuccess)
                re = read_split_probe(times.data(), ctas);
            if (re != cudaSuccess) {
                st = cuda_failed(re);
                break;
            }
            unsigned long long t0 = times[0];
            for (int c = 1; c < ctas; ++c)
                t0 = times[2 * c] < t0 ? times[2 * c] : t0;
            for (int c = 0; c < ctas; ++c) {
                S[c] += static_cast<double>(times[2 * c] - t0) / kCallsPerRound;
                F[c] += static_cast<double>(times[2 * c + 1] > t0 ? times[2 * c + 1] - t0 : 0) / kCallsPerRound;
            }
        }
        if (st != PKV_OK)
            break;
        // Each CTA streams its share at rate w_c / (F_c - S_c); for all to
        // finish together at the mean finish time its new share is that rate
        // times (mean F - S_c).  Normalised to the middle of the weight range.
        double fbar = 0.0;
        for (int c = 0; c < ctas; ++c)
            fbar += F[c] / ctas;
        std::vector<double> nw(static_cast<size_t>(ctas), kMean);
        double sum = 0.0;
        for (int c = 0; c < ctas; ++c) {
            const double busy = F[c] - S[c], left = fbar - S[c];
            nw[c] = (busy > 0.0 && left > 0.0) ? w[c] * left / busy : w[c];
            sum += nw[c];
        }
        for (int c = 0; c < ctas; ++c) {
            wd[c] = sum > 0.0 ? nw[c] * kMean * ctas / sum : kMean;
            w[c] = quantise(wd[c]);
        }
        // The first round moves the weights from equal to near the balance;
        // later rounds estimate the same balance again, and their average
        // (not their last) is kept, so one call's timing noise does not.
        if (r > 0 || rounds == 1) {
            for (int c = 0; c < ctas; ++c)
                avg[c] += wd[c];
            ++n_avg;
        }
        st = set_split(w.data(), ctas);
    }
    if (st == PKV_OK && n_avg > 0) {
        double sum = 0.0;
        for (int c = 0; c < ctas; ++c)
            sum += avg[c];
        for (int c = 0; c < ctas; ++c)
            w[c] = quantise(sum > 0.0 ? avg[c] * kMean * ctas / sum : kMean);
        st = set_split(w.data(), ctas);
    }
    if (st != PKV_OK) {
        set_split(nullptr, 0);
        return st;
    }
    if (n_out)
        *n_out = ctas;
    if (weights_out) {
        if (capacity < ctas)
            return PKV_ERR_SHAPE;
        for (int c = 0; c < ctas; ++c)
            weights_out[c] = w[c];
    }
    return PKV_OK;
}

size_t pkv_prefill_workspace_size(int batch, int num_kv_heads, int max_kv_len, int64_t max_total_kv)
{
    if (batch < 0 || num_kv_heads <= 0 || max_kv_len < 0 || max_total_kv < 0)
        return 0;
    return prefill_workspace_bytes(batch, num_kv_heads, max_kv_len, max_total_kv);
}

pkv_status pkv_paged_prefill(const void *q, const int32_t *cu_q, int total_q, int max_q_len, const uint8_t *k_cache,
                             const uint8_t *v_cache, const float *k_scale, const float *v_scale,
                             const int32_t *block_table, int max_pages_per_seq, const int32_t *seq_lens,
                             const int32_t *seq_page_sizes, int batch, int max_kv_len, int64_t max_total_kv,
                             int num_q_heads, int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
                             float sm_scale, void *out, int out_dtype, void *workspace, size_t workspace_bytes,
                             int32_t *device_error, cudaStream_t stream)
{
    pkv_status st = check_decode_shape(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_seq,
                                       num_pages);
    if (st != PKV_OK)
        return st;
    if (total_q < 0 || max_q_len < 0 || max_kv_len < 0 || max_total_kv < 0)
        return PKV_ERR_SHAPE;
    if (out_dtype != PKV_F32 && out_dtype != PKV_BF16)
        return PKV_ERR_DTYPE;
    if (!(sm_scale > 0.f) || isinf(sm_scale))            // the kernel scales raw scores after their maximum
        return PKV_ERR_SHAPE;
    if (seq_page_sizes && static_cast<int64_t>(max_pages_per_seq) * 256 >= (int64_t(1) << 31))
        return PKV_ERR_UNSUPPORTED;
    if (batch == 0 || total_q == 0 || max_q_len == 0)
        return PKV_OK;
    if (!q || !cu_q || !k_cache || !v_cache || !k_scale || !v_scale || !block_table || !seq_lens || !out)
        return PKV_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(cu_q, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(k_scale, 4) ||
        !aligned(v_scale, 4) || !aligned(device_error, 4) || !aligned(seq_page_sizes, 4))
        return PKV_ERR_ALIGN;
    const int group = num_q_heads / num_kv_heads;
    const int tpt = 128 / group;
    const int64_t max_tiles = (static_cast<int64_t>(max_q_len) + tpt - 1) / tpt;
    if (static_cast<int64_t>(batch) * num_kv_heads * max_tiles >= (int64_t(1) << 31))
        return PKV_ERR_UNSUPPORTED;
    if (max_kv_len == 0)
        return PKV_OK;                                   // no sequence can hold a query
    const long long rows = prefill_rows_bound(batch, num_kv_heads, max_kv_len, max_total_kv);
    if (rows >= (int64_t(1) << 31) || batch + 1 + 8 > 49152)
        return PKV_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < prefill_workspace_bytes(batch, num_kv_heads, max_kv_len, max_total_kv))
        return PKV_ERR_WORKSPACE;
    int *tile_off = static_cast<int *>(workspace);
    __half *k16 = reinterpret_cast<__half *>(static_cast<uint8_t *>(workspace) + prefill_header_bytes(batch));
    __half *v16 = k16 + static_cast<size_t>(rows) * kHeadDim;

    alignas(64) CUtensorMap tm_q;
    alignas(64) CUtensorMap tm_k;
    alignas(64) CUtensorMap tm_v;
    if (!make_q_map(&tm_q, q, total_q, num_q_heads, group, tpt) ||
        !make_kv16_map(&tm_k, k16, rows, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) ||
        !make_kv16_map(&tm_v, v16, rows, CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
        return cuda_failed(cudaErrorInvalidValue);

    PrefillArgs a;
    a.cu_q = cu_q;
    a.total_q = total_q;
    a.max_q_len = max_q_len;
    a.tokens_per_tile = tpt;
    a.max_tiles = static_cast<int>(max_tiles);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_table = block_table;
    a.max_pages = max_pages_per_seq;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.hq = num_q_heads;
    a.hkv = num_kv_heads;
    a.group = group;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.page_sizes = seq_page_sizes;
    a.pool_log2 = 31 - __builtin_clz(static_cast<unsigned>(page_size));
    a.max_kv_len = max_kv_len;
    a.tile_off = tile_off;
    a.rows_cap = rows;
    a.k16 = k16;
    a.v16 = v16;
    // Test facility for the timeout path (pkv_test_withhold_load): that CTA
    // never loads its first K tile, so its MMA warp's wait runs out.
    a.withhold_block = g_withhold.load(std::memory_order_relaxed);
    a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
    a.out = out;
    a.out_f32 = out_dtype == PKV_F32;
    a.err = device_error;
    const cudaError_t e = launch_paged_prefill(a, tm_q, tm_k, tm_v, stream);
    return e == cudaSuccess ? PKV_OK : cuda_failed(e);
}

}  // extern "C"
