// pkv_paged_gqa_decode_noalloc: the decode call for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc at all: a serving engine that reserves
// all device memory up front and hands out only its own pool, a plugin
// running inside another runtime whose allocator it must not bypass, or a
// latency-critical loop that cannot afford an allocation's implicit
// synchronisation.  Such a caller also cannot easily keep a per-call
// workspace alive.  This entry point takes the same inputs and outputs as
// pkv_paged_gqa_decode but keeps its split-K scratch in a fixed-size array
// that is part of the library image itself, so the call needs no workspace
// and performs no allocation.
//
// Costs and rules of that choice:
//   * every GPU on which the library is loaded holds the array (kNoAllocScratchBytes)
//     until the process exits;
//   * all calls share it: two calls that overlap on the GPU (different streams,
//     or different host threads without ordering) race on it and give wrong
//     results.  Calls on one stream are ordered and safe.
//   * it keeps the last call's contents; the decode writes every value it
//     later reads, so nothing needs clearing between calls;
//   * sizes whose scratch would exceed the array are rejected with
//     PKV_ERR_WORKSPACE.
//
// The first call on each device looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and caches it; make that
// first call before any stream capture begins.  The cache is keyed by the
// device's current context, so after cudaDeviceReset (which destroys the
// context and unloads the library's device image) the next call on that
// device looks the address up again instead of using a stale one.
#include <algorithm>
#include <mutex>

#include "context.h"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

// Host code must not take this symbol's address as a device pointer: on the
// host it names a stand-in object.  The device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct ScratchEntry {
    unsigned long long ctx_id = 0;   // context the address belongs to (0: none yet)
    void *ptr = nullptr;
};

std::mutex g_noalloc_mu;
ScratchEntry g_noalloc[64];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name)
{
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(fn);
}

void *scratch_for_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    ScratchEntry &e = g_noalloc[dev];
    unsigned long long id = 0;
    if (e.ptr != nullptr && pkv::current_context_id(&id) && id == e.ctx_id)
        return e.ptr;
    // Set-up for this device (or its new context): the lookup also makes the
    // device's primary context current if it was not yet.
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !pkv::current_context_id(&id))
        return nullptr;
    e.ptr = p;
    e.ctx_id = id;
    return p;
}

}  // namespace

bool pkv::current_context_id(unsigned long long *id)
{
    // function-local statics: looked up once, thread-safely
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    CUcontext ctx = nullptr;
    return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
           get_id(ctx, id) == CUDA_SUCCESS;
}

extern "C" size_t pkv_decode_noalloc_scratch_bytes(void)
{
    return kNoAllocScratchBytes;
}

extern "C" pkv_status pkv_paged_gqa_decode_noalloc(
    const void *q, const uint8_t *k_cache, const uint8_t *v_cache, const float *k_scale, const float *v_scale,
    const int32_t *block_table, int max_pages_per_seq, const int32_t *seq_lens, int max_seq_len,
    const int32_t *seq_page_sizes, int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
    int64_t num_pages, float sm_scale, void *out, int out_dtype, int32_t *device_error, int max_ctas,
    cudaStream_t stream)
{
    auto full_check = [&]() {   // sizes the library rejects anyway: let the full check report the reason
        return pkv_paged_gqa_decode(q, k_cache, v_cache, k_scale, v_scale, block_table, max_pages_per_seq, seq_lens,
                                    max_seq_len, seq_page_sizes, batch, num_q_heads, num_kv_heads, head_dim, page_size,
                                    num_pages, sm_scale, out, out_dtype, nullptr, 0, device_error, max_ctas, stream);
    };
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        max_pages_per_seq <= 0 || max_seq_len < 0)
        return full_check();
    const int bound = max_seq_len > 0 ? max_seq_len
                      : static_cast<int>(std::min<int64_t>(static_cast<int64_t>(max_pages_per_seq) * page_size,
                                                           INT32_MAX));
    const size_t need =
        pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, bound, page_size, max_ctas);
    if (need == 0)
        return full_check();
    if (need > kNoAllocScratchBytes)
        return PKV_ERR_WORKSPACE;
    void *scratch = scratch_for_current_device();
    if (!scratch)
        return PKV_ERR_CUDA;
    return pkv_paged_gqa_decode(q, k_cache, v_cache, k_scale, v_scale, block_table, max_pages_per_seq, seq_lens,
                                bound, seq_page_sizes, batch, num_q_heads, num_kv_heads, head_dim, page_size,
                                num_pages, sm_scale, out, out_dtype, scratch, kNoAllocScratchBytes, device_error,
                                max_ctas, stream);
}
