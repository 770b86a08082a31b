// paged_prefill: chunked-prefill attention over the paged FP8 KV cache, on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes.  A long prompt is prefilled in chunks and each chunk's KV
// joins the cache before its queries attend (0539edu.com Llama 3 notes, §2.2:
// a 128K prompt as 8 chunks of 16K).  Sequence b brings a chunk of n_b
// queries; query c sits at position L_b - n_b + c and, for each query head i,
// attends to the cached tokens 0 .. L_b - n_b + c of kv head i / G (GQA,
// "FP8量化与长上下文实测：Llama 3 70B部署优化指南" §1.2), with K and V read as
// E4M3 value x per-(kv head) scale (same guide, §3.1-§3.2).  The chunk's own
// K/V are already in the pages (kv_append_fp8 ran first).
//
// Two launches.
//   kv_widen_kernel    reads every cached token the chunk can see once from
//                      the pages (block-table lookup) and writes it widened
//                      (exactly: E4M3 has 3 mantissa bits) to dense
//                      per-(sequence, kv head) copies in the caller's
//                      workspace, K as bf16 and V as f16, zero rows up to the
//                      next 128-key tile.  HBM-bound, about 1/1000 of the
//                      attention time.
//   paged_prefill_kernel  one CTA per (sequence, kv head, tile of 128 / G query
//                      tokens).  The tile's 128 rows are (token, query head of
//                      the group) pairs, so each K/V tile brought on chip
//                      serves all G heads.  Keys are visited in tiles of 128.
// Widening once, instead of in every CTA that reads a tile (a key tile of a
// 16K chunk is read by about a thousand CTAs), takes the FP8 conversions off
// the attention kernel's critical resources and turns 16 page-sized copies
// per tile into 4 tile-sized ones.
//
// Attention kernel roles (one per warp):
//   warp 0      TMA: the bf16 query tile (once; it stays in shared memory as
//               the A operand of S = Q K^T), then per key tile two 16 KB boxes
//               of K and two of V, already in the 128B-swizzled operand
//               layout, into 2- and 3-stage rings;
//   warp 1      owns the 512 TMEM columns and issues tcgen05.mma (the warp
//               runs the loop converged, one elected lane issues; a loop run
//               by a lone lane made every MMA issue compete with the softmax
//               warps of its SMSP and left the tensor pipe half idle):
//                 S_j   = Q K_j^T  M 128 rows, N 128 keys, K 128 dims, bf16;
//                                  S in TMEM (2 buffers, so S_{j+1} overlaps
//                                  softmax j)
//                 O_seg += P_j V_j A = P_j read from TMEM (f16 hi + lo parts),
//                                  B = V_j stored N(=dim)-major
//   warps 2-9   online softmax, two warps per TMEM lane quarter: one row per
//               thread, each warp one half (64 keys) of the tile.  The row
//               maximum is exchanged through shared memory; exp2 domain, lazy
//               rescaling (only when the maximum grows by more than 2^8);
//               P is written over S in TMEM.  Every kFold key tiles they add
//               O_seg into O (a second TMEM accumulator) in fp32 and the next
//               PV starts O_seg afresh, so no chain of accumulating MMAs is
//               longer than 16 kFold; at the end each warp stores its half of
//               (O + O_seg) / l x v_scale.
// Every wait is bounded (2 s): on expiry the CTA sets PKV_DEVERR_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and exits.
#include <mutex>

#include "context.h"
#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;                       // M: rows of a query tile
constexpr int kKeys = 128;                       // keys per tile
constexpr int kKStages = 2, kVStages = 3;        // operand rings: K bf16, V f16
constexpr int kFold = 32;                        // key tiles per tensor-core accumulation segment of O
constexpr int kSmWarp0 = 2;                      // first softmax warp
constexpr int kSmWarps = 8;
constexpr int kPThreads = 32 * (kSmWarp0 + kSmWarps);
constexpr uint32_t kColO = 256, kColM = 384;     // TMEM columns: S/P 0-255, O of the segment 256-383, O 384-511
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr unsigned kAll = 0xffffffffu;
static_assert(kSmWarps == 8, "two softmax warps per TMEM lane quarter");

// Shared memory, offsets from a 1024-byte aligned base.  Operand tiles are
// [2 column blocks][128 rows][128 bytes] with the 128-byte swizzle.
struct PS {
    static constexpr int kTile = 32768;
    static constexpr int kQ = 0;                           // the query tile (bf16)
    static constexpr int kK16 = kQ + kTile;                // kKStages tiles (bf16)
    static constexpr int kV16 = kK16 + kKStages * kTile;   // kVStages tiles (f16)
    static constexpr int kRedMax = kV16 + kVStages * kTile;   // float [2 parities][2 halves][128 rows]
    static constexpr int kRedL = kRedMax + 2048;              // float [2 halves][128 rows]
    static constexpr int kBars = kRedL + 1024;
    enum {
        Q_FULL, Q_READY, K_FULL, K_EMPTY = K_FULL + kKStages, V_FULL = K_EMPTY + kKStages,
        V_EMPTY = V_FULL + kVStages, S_FULL = V_EMPTY + kVStages, P_FULL = S_FULL + 2, PV_DONE = P_FULL + 2,
        O_FINAL, DRAIN,
        MX = DRAIN + 1,                                  // [2 tile parities][4 lane quarters]: row-max exchange
        LX = MX + 8,                                     // [4 lane quarters]: final row-sum exchange
        kNumBars = LX + 4
    };
    static constexpr int kTmem = kBars + kNumBars * 8;
    static constexpr int kFlag = kTmem + 4;
    static constexpr int kEnd = kFlag + 4;
    static constexpr size_t bytes() { return static_cast<size_t>(kEnd) + 1024; }
};
static_assert(PS::bytes() <= 232448, "prefill tile buffers exceed the shared memory of one CTA");

// Bounded wait, one thread.  honour_abort = false for drains.
__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int32_t *err,
                                      bool honour_abort = true)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 15u) == 0) {
            if (honour_abort && *abort_flag)
                return false;
            if (global_timer_ns() - t0 > kWaitNs) {
                *abort_flag = 1;
                if (err)
                    atomicOr(err, PKV_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait by a whole warp; the result is warp-uniform.
__device__ __forceinline__ bool wwait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int32_t *err,
                                      int lane)
{
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (__all_sync(kAll, mbar_try_wait(bar, parity)))
            return true;
        if ((it & 15u) == 15u) {
            int stop = 0;
            if (lane == 0) {
                if (*abort_flag) {
                    stop = 1;
                } else if (t0 == 0) {
                    t0 = global_timer_ns();
                } else if (global_timer_ns() - t0 > kWaitNs) {
                    *abort_flag = 1;
                    if (err)
                        atomicOr(err, PKV_DEVERR_TIMEOUT);
                    stop = 1;
                }
            }
            if (__shfl_sync(kAll, stop, 0))
                return false;
        }
    }
}

// Descriptors are built once per ring stage; a K step then only advances the
// start-address field (bytes / 16, the low bits of the descriptor), so the
// issuing thread spends its time issuing, not rebuilding 64-bit descriptors.
// K-major operand (128 rows x 128 dims, 128B swizzle; the query tile as A and
// a K tile as B of S = Q K^T): K step s of 16 dims starts (s / 4) * 16 KB +
// (s % 4) * 32 B into the tile.
__device__ __forceinline__ uint64_t kmajor_base(uint32_t tile)
{
    return tc::smem_desc_sw128(tile, 16, 1024);
}
__device__ __forceinline__ uint64_t kmajor_step(uint64_t base, int s)
{
    return base + static_cast<uint64_t>(((s >> 2) * 16384 + (s & 3) * 32) >> 4);
}

// V as the B operand of O += P V: rows = keys (the K dimension), 128 dims (N)
// contiguous in two 64-dim column blocks 16 KB apart; K step s = keys 16s..16s+15
// starts s * 2 KB into the tile.
__device__ __forceinline__ uint64_t vmn_base(uint32_t tile)
{
    return tc::smem_desc_sw128(tile, 16384, 1024);
}
__device__ __forceinline__ uint64_t vmn_step(uint64_t base, int s)
{
    return base + static_cast<uint64_t>((s * 2048) >> 4);
}

// f16 pair -> bf16 pair (exact for widened E4M3 values: 3 mantissa bits).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h)
{
    const float2 f = f16x2_to_f32x2(h);
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<uint32_t *>(&b);
}

// P = 2^(x - m) as two f16 parts: hi = P with its low 13 mantissa bits cleared
// (exact in f16 for P >= 2^-14), lo = the rest (exact in fp32, rounded to f16).
// hi + lo equals P to about 2^-22 relative; below 2^-14 the parts keep an
// absolute error under 2^-24.
__device__ __forceinline__ void split_pair(float p0, float p1, uint32_t &hi, uint32_t &lo)
{
    const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
    const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
    hi = f32x2_to_f16x2(h0, h1);
    lo = f32x2_to_f16x2(p0 - h0, p1 - h1);
}

// Packed pairs of fp32 (one 64-bit register pair): the paired add and fma
// run two lanes of fp32 arithmetic per instruction, each rounded exactly as
// the scalar operation, so results equal the scalar code bit for bit.
__device__ __forceinline__ uint64_t f2_pack(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float2 f2_unpack(uint64_t r)
{
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// max(a, b, c) in one instruction (exact, like two fmaxf).
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// True in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one()
{
    uint32_t p;
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, e;\n\t}"
        : "=r"(p));
    return p != 0;
}

// Checks a sequence's sizes; false (and PKV_DEVERR_SEQLEN when `report`) when
// the chunk or its length are inconsistent.
__device__ __forceinline__ bool sequence_ok(const PrefillArgs &a, int b, int q0, int q1, int L, bool report)
{
    const int n = q1 - q0;
    const int lp = seq_page_log2(a, b);
    const bool ok = q0 >= 0 && n >= 0 && q1 <= a.total_q && n <= a.max_q_len && L >= n && L <= a.max_kv_len &&
                    lp >= 0 && static_cast<int64_t>(L) <= (static_cast<int64_t>(a.max_pages) << lp);
    if (!ok && report && a.err)
        atomicOr(a.err, lp < 0 ? PKV_DEVERR_PAGESIZE : PKV_DEVERR_SEQLEN);
    return ok;
}

// 128-row tiles of sequence b's widened region (all its kv heads): zero for a
// sequence with an empty or inconsistent chunk.
__device__ __forceinline__ long long region_tiles(const PrefillArgs &a, int b)
{
    const int q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1);
    const int L = __ldg(a.seq_lens + b);
    if (q1 - q0 <= 0 || !sequence_ok(a, b, q0, q1, L, false))
        return 0;
    return static_cast<long long>(a.hkv) * ((L + kKeys - 1) / kKeys);
}

// ---------------------------------------------------------------------- widening
// Every CTA first lays out the regions: tile_off[b] = the first 128-row tile
// of sequence b's region, a prefix sum of region_tiles (saturated just past
// the workspace's capacity, so a region that does not fit is recognisable);
// CTA 0 also stores them for the attention kernel and flags sequences whose
// region does not fit.  Then one thread per 16 FP8 bytes (16 dims of one key
// row of one kv head) of K and of V reads them through the block table and
// writes 32 bytes of 16-bit values to the region.  Rows from L up to the next
// multiple of 128 are zeros.
__global__ void __launch_bounds__(256) kv_widen_kernel(const PrefillArgs a)
{
    extern __shared__ int off[];                         // [batch + 1], then 8 warp sums
    int *warp_sum = off + a.batch + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long cap_tiles = a.rows_cap / 128;
    {
        const int chunk = (a.batch + 255) / 256;
        const int b0 = min(a.batch, tid * chunk), b1 = min(a.batch, b0 + chunk);
        long long local = 0;
        for (int b = b0; b < b1; ++b)
            local += region_tiles(a, b);
        // saturate: nothing past cap_tiles + 1 matters
        int loc = static_cast<int>(local < cap_tiles + 1 ? local : cap_tiles + 1);
        int incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kAll, incl, o);
            if (lane >= o)
                incl = min(incl + v, static_cast<int>(cap_tiles + 1));
        }
        if (lane == 31)
            warp_sum[warp] = incl;
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w)
            base = min(base + warp_sum[w], static_cast<int>(cap_tiles + 1));
        int run = min(base + incl - loc, static_cast<int>(cap_tiles + 1));
        for (int b = b0; b < b1; ++b) {
            off[b] = run;
            run = static_cast<int>(min(run + region_tiles(a, b), cap_tiles + 1));
        }
        if (tid == 255)
            off[a.batch] = min(base + incl, static_cast<int>(cap_tiles + 1));
        __syncthreads();
        if (blockIdx.x == 0) {
            for (int b = tid; b <= a.batch; b += 256) {
                a.tile_off[b] = off[b];
                if (b < a.batch && off[b + 1] > cap_tiles && off[b + 1] > off[b] && a.err)
                    atomicOr(a.err, PKV_DEVERR_SEQLEN);          // its region does not fit the workspace
            }
        }
    }
    const int64_t end_tile = min(static_cast<long long>(off[a.batch]), cap_tiles);
    const int64_t total = end_tile * 128 * 8;
    for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < total;
         u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t R = u >> 3;                               // row of the copies
        const int e = static_cast<int>(u & 7);                  // dims 16 e .. 16 e + 15
        const int tile = static_cast<int>(R >> 7);
        int lo = 0, hi = a.batch - 1;                           // the sequence whose region holds the tile
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (off[mid] <= tile)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int b = lo;
        if (off[b + 1] > cap_tiles)
            continue;                                           // region past the workspace: flagged above
        const int L = __ldg(a.seq_lens + b);
        const int pad = ((L + kKeys - 1) / kKeys) * kKeys;
        const int local = static_cast<int>(R - static_cast<int64_t>(off[b]) * 128);
        const int h = local / pad, r = local - h * pad;
        uint4 k = make_uint4(0, 0, 0, 0), v = make_uint4(0, 0, 0, 0);
        if (r < L) {
            int pg, row;
            if (seq_token_page(a, b, seq_page_log2(a, b), r, pg, row)) {
                const int64_t src = ((static_cast<int64_t>(pg) * a.hkv + h) * a.page_size + row) * kHeadDim + 16 * e;
                k = __ldg(reinterpret_cast<const uint4 *>(a.k_cache + src));
                v = __ldg(reinterpret_cast<const uint4 *>(a.v_cache + src));
            } else if (e == 0 && a.err) {
                atomicOr(a.err, PKV_DEVERR_PAGE);
            }
        }
        const int64_t dst = R * kHeadDim + 16 * e;              // in 16-bit elements
        uint4 lo4, hi4;
        e4m3x4_to_f16x4(k.x, lo4.x, lo4.y);
        e4m3x4_to_f16x4(k.y, lo4.z, lo4.w);
        e4m3x4_to_f16x4(k.z, hi4.x, hi4.y);
        e4m3x4_to_f16x4(k.w, hi4.z, hi4.w);
        reinterpret_cast<uint4 *>(a.k16 + dst)[0] = make_uint4(f16x2_to_bf16x2(lo4.x), f16x2_to_bf16x2(lo4.y),
                                                               f16x2_to_bf16x2(lo4.z), f16x2_to_bf16x2(lo4.w));
        reinterpret_cast<uint4 *>(a.k16 + dst)[1] = make_uint4(f16x2_to_bf16x2(hi4.x), f16x2_to_bf16x2(hi4.y),
                                                               f16x2_to_bf16x2(hi4.z), f16x2_to_bf16x2(hi4.w));
        e4m3x4_to_f16x4(v.x, lo4.x, lo4.y);
        e4m3x4_to_f16x4(v.y, lo4.z, lo4.w);
        e4m3x4_to_f16x4(v.z, hi4.x, hi4.y);
        e4m3x4_to_f16x4(v.w, hi4.z, hi4.w);
        reinterpret_cast<uint4 *>(a.v16 + dst)[0] = lo4;
        reinterpret_cast<uint4 *>(a.v16 + dst)[1] = hi4;
    }
}

// ---------------------------------------------------------------------- attention
__global__ void __launch_bounds__(kPThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a)
{
    // ---------------------------------------------------------------- the tile
    // (sequence, kv head)-major order, heaviest query tiles (largest positions)
    // first within each: the CTAs resident at one time mostly read the K/V of
    // one kv head, so the tiles they share stay in L2.
    const int bh = blockIdx.x / a.max_tiles;
    const int rank = blockIdx.x - bh * a.max_tiles;
    const int qt = a.max_tiles - 1 - rank;
    const int b = bh / a.hkv;
    const int h = bh - b * a.hkv;
    const int G = a.group, tpt = a.tokens_per_tile;
    const int q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1);
    const int n = q1 - q0;
    const int L = __ldg(a.seq_lens + b);
    if (!sequence_ok(a, b, q0, q1, L, qt == 0 && h == 0 && threadIdx.x == 0))
        return;
    // this sequence's widened region (laid out by the widening kernel); a
    // region past the workspace was flagged there and is not attended
    const int off0 = __ldg(a.tile_off + b), off1 = __ldg(a.tile_off + b + 1);
    if (off1 > a.rows_cap / 128 || off1 - off0 != a.hkv * ((L + kKeys - 1) / kKeys))
        return;
    const int row0 = off0 * 128 + h * (off1 - off0) / a.hkv * 128;   // first row of this kv head's copy
    const int t0 = qt * tpt;                             // first token of the tile in the chunk
    if (t0 >= n)
        return;
    const int nv = min(tpt, n - t0);                     // tokens of the tile
    const int pos0 = L - n + t0;                         // position of its first token
    const int last = pos0 + nv - 1;                      // largest position in the tile
    const int nt = last / kKeys + 1;                     // key tiles to visit

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(smem);
    auto bar = [&](int i) { return sb + PS::kBars + 8u * i; };
    uint64_t *bar_ptr = reinterpret_cast<uint64_t *>(smem + PS::kBars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + PS::kTmem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + PS::kFlag);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(PS::Q_FULL), 1);
        mbar_init(bar(PS::Q_READY), kSmWarps);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(bar(PS::K_FULL + i), 1);
            mbar_init(bar(PS::K_EMPTY + i), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(bar(PS::V_FULL + i), 1);
            mbar_init(bar(PS::V_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(PS::S_FULL + i), 1);
            mbar_init(bar(PS::P_FULL + i), 32 * kSmWarps);
        }
        mbar_init(bar(PS::PV_DONE), 1);
        mbar_init(bar(PS::O_FINAL), 1);
        mbar_init(bar(PS::DRAIN), 1);
        for (int i = 0; i < 8; ++i)
            mbar_init(bar(PS::MX + i), 64);
        for (int i = 0; i < 4; ++i)
            mbar_init(bar(PS::LX + i), 64);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tslot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA: query tile, f16 K/V tiles
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            mbar_arrive_expect_tx(bar(PS::Q_FULL), 2u * 128u * G * tpt);
            const uint64_t pol = l2_policy_evict_first();
            tma_load_3d(sb + PS::kQ, &tm_q, 0, h * G, q0 + t0, bar(PS::Q_FULL), pol);
            tma_load_3d(sb + PS::kQ + 16384, &tm_q, 64, h * G, q0 + t0, bar(PS::Q_FULL), pol);
            const int z = 0;
            uint32_t karmed[kKStages] = {}, varmed[kVStages] = {};
            bool ok = true;
            for (int t = 0; ok && t < nt; ++t) {
                const int ks = t % kKStages, vs = t % kVStages;
                if (t >= kKStages &&
                    !pwait(bar(PS::K_EMPTY + ks), ((t / kKStages) - 1) & 1, abort_flag, a.err)) {
                    ok = false;
                    break;
                }
                // (test facility: the withheld CTA never arms or loads its first K tile)
                if (t > 0 || static_cast<int>(blockIdx.x) != a.withhold_block) {
                    mbar_arrive_expect_tx(bar(PS::K_FULL + ks), PS::kTile);
                    karmed[ks] = static_cast<uint32_t>(t / kKStages) + 1;
                    tma_load_3d_plain(sb + PS::kK16 + ks * PS::kTile, &tm_k, 0, row0 + t * kKeys, z,
                                      bar(PS::K_FULL + ks));
                    tma_load_3d_plain(sb + PS::kK16 + ks * PS::kTile + 16384, &tm_k, 64, row0 + t * kKeys, z,
                                      bar(PS::K_FULL + ks));
                }
                if (t >= kVStages &&
                    !pwait(bar(PS::V_EMPTY + vs), ((t / kVStages) - 1) & 1, abort_flag, a.err)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(PS::V_FULL + vs), PS::kTile);
                varmed[vs] = static_cast<uint32_t>(t / kVStages) + 1;
                tma_load_3d_plain(sb + PS::kV16 + vs * PS::kTile, &tm_v, 0, row0 + t * kKeys, z,
                                  bar(PS::V_FULL + vs));
                tma_load_3d_plain(sb + PS::kV16 + vs * PS::kTile + 16384, &tm_v, 64, row0 + t * kKeys, z,
                                  bar(PS::V_FULL + vs));
            }
            // No copy may still be landing when the CTA leaves.
            pwait(bar(PS::Q_FULL), 0, abort_flag, a.err, false);
            for (int s = 0; s < kKStages; ++s)
                if (karmed[s])
                    pwait(bar(PS::K_FULL + s), (karmed[s] - 1) & 1, abort_flag, a.err, false);
            for (int s = 0; s < kVStages; ++s)
                if (varmed[s])
                    pwait(bar(PS::V_FULL + s), (varmed[s] - 1) & 1, abort_flag, a.err, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        // The whole warp runs this loop converged (descriptors stay warp-uniform);
        // one elected lane issues the MMAs and the commits that track them.
        const uint32_t id_qk = tc::idesc_bf16_f32(kRows, kKeys, false);
        const uint32_t id_pv = tc::idesc_f16_f32(kRows, kHeadDim, true);
        const uint32_t o_tm = tm + kColO;
        const uint64_t qdesc = kmajor_base(sb + PS::kQ);
        uint64_t kdesc[kKStages], vdesc[kVStages];
#pragma unroll
        for (int i = 0; i < kKStages; ++i)
            kdesc[i] = kmajor_base(sb + PS::kK16 + i * PS::kTile);
#pragma unroll
        for (int i = 0; i < kVStages; ++i)
            vdesc[i] = vmn_base(sb + PS::kV16 + i * PS::kTile);
        const bool leader = elect_one();
        bool ok = wwait(bar(PS::Q_READY), 0, abort_flag, a.err, lane);
        tc::fence_after();
        for (int j = 0; ok && j <= nt; ++j) {
            if (j < nt) {
                const int fb = j & 1, ks = j % kKStages;
                if (!wwait(bar(PS::K_FULL + ks), (j / kKStages) & 1, abort_flag, a.err, lane)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint64_t kd = kdesc[ks];
                const uint32_t s_tm = tm + fb * 128;
                if (leader) {
#pragma unroll
                    for (int s = 0; s < 8; ++s)         // dims 16s..16s+15
                        tc::mma_ss(s_tm, kmajor_step(qdesc, s), kmajor_step(kd, s), id_qk, s > 0);
                    tc::commit(bar_ptr + PS::S_FULL + fb);
                    tc::commit(bar_ptr + PS::K_EMPTY + ks);
                }
                __syncwarp();
            }
            if (j > 0) {
                const int i = j - 1, fb = i & 1, vs = i % kVStages;
                if (!wwait(bar(PS::P_FULL + fb), (i >> 1) & 1, abort_flag, a.err, lane) ||
                    !wwait(bar(PS::V_FULL + vs), (i / kVStages) & 1, abort_flag, a.err, lane)) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                const uint64_t vd = vdesc[vs];
                const uint32_t p_tm = tm + fb * 128;
                const uint32_t acc0 = (i % kFold) != 0 ? 1u : 0u;   // a new segment starts from zero
                if (leader) {
                    // keys 16s..16s+15: hi parts in columns 32(s/2) + 8(s%2) .. +7, lo 16 further
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_ts(o_tm, p_tm + 32 * (s >> 1) + 8 * (s & 1), vmn_step(vd, s), id_pv,
                                   s > 0 ? 1u : acc0);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_ts(o_tm, p_tm + 32 * (s >> 1) + 8 * (s & 1) + 16, vmn_step(vd, s), id_pv, 1u);
                    tc::commit(bar_ptr + PS::PV_DONE);
                    tc::commit(bar_ptr + PS::V_EMPTY + vs);
                    if (i == nt - 1)
                        tc::commit(bar_ptr + PS::O_FINAL);
                }
                __syncwarp();
            }
        }
        // Every MMA issued has finished before TMEM is released.
        if (leader) {
            tc::commit(bar_ptr + PS::DRAIN);
            pwait(bar(PS::DRAIN), 0, abort_flag, a.err, false);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + output
        const int qtr = warp & 3;                        // TMEM lane quarter of this warp
        const int half = (warp - kSmWarp0) >> 2;         // keys 64 half .. 64 half + 63 of every tile
        const int row = qtr * 32 + lane;
        const int tl = row / G;
        const int g = row - tl * G;
        const bool valid = row < G * tpt && tl < nv;
        const int p_row = valid ? pos0 + tl : last;      // padding rows mirror the last row
        const float sl2 = __ldg(a.k_scale + h) * a.sm_scale_log2;
        const uint32_t lanes = tm + (static_cast<uint32_t>(qtr * 32) << 16);
        float *red_max = reinterpret_cast<float *>(smem + PS::kRedMax);
        float *red_l = reinterpret_cast<float *>(smem + PS::kRedL);
        float m = -INFINITY, l = 0.f;
        // The query tile is the A operand of S = Q K^T as TMA wrote it (bf16,
        // 128B-swizzled, row = token x G + head).  Rows past the G x tpt the
        // copy fills are zeroed here (this warp: its row, dims 64 half ..).
        bool ok = wwait(bar(PS::Q_FULL), 0, abort_flag, a.err, lane);
        if (ok) {
            if (row >= G * tpt) {
                uint4 *qrow = reinterpret_cast<uint4 *>(smem + PS::kQ + half * 16384 + row * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    qrow[c] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();     // generic-proxy writes -> visible to the tensor cores
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(PS::Q_READY));
        }
        for (int j = 0; ok && j < nt; ++j) {
            const int fb = j & 1;
            if (!wwait(bar(PS::S_FULL + fb), (j >> 1) & 1, abort_flag, a.err, lane)) {
                ok = false;
                break;
            }
            tc::fence_after();
            const uint32_t s_tm = lanes + fb * 128 + 64 * half;
            uint32_t x[2][32];
            tc::ld32(s_tm, x[0]);
            tc::ld32(s_tm + 32, x[1]);
            tc::wait_ld();
            // pass 1 on the raw scores (sl2 > 0): the maximum of the visible scaled
            // logits of this half is sl2 x the maximum raw score.  Hidden keys
            // become -inf, so pass 2 needs no mask.
            const int vis = p_row - j * kKeys - 64 * half;
            float mx[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mx[k] = -INFINITY;
            if (vis < 63) {
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        if (32 * c + k > vis)
                            x[c][k] = __float_as_uint(-INFINITY);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int k = 0; k < 32; k += 2)
                    mx[(k >> 1) & 7] = max3(mx[(k >> 1) & 7], __uint_as_float(x[c][k]), __uint_as_float(x[c][k + 1]));
            const float mh = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
            // P = 2^(x sl2 - mm) <= 2^8 as f16 hi + lo, written over each 32-column
            // piece of S (hi in its first 16 columns, lo in the last 16); returns
            // the half row's sum of P.
            // Pairs of elements go through the paired fp32 add / fma (fewer
            // instructions on the softmax warps' issue slots; same roundings).
            auto emit = [&](float mm) -> float {
                uint64_t ls[4];                            // ls[i] = sums of elements 2i, 2i+1 (mod 8)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    ls[k] = 0ull;
                const uint64_t sl2x2 = f2_pack(sl2, sl2), nmm = f2_pack(-mm, -mm);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t ph[16], pl[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const float2 y = f2_unpack(
                            f2_fma(f2_pack(__uint_as_float(x[c][2 * q]), __uint_as_float(x[c][2 * q + 1])), sl2x2, nmm));
                        const float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
                        const uint64_t pp = f2_pack(p0, p1);
                        ls[q & 3] = f2_add(ls[q & 3], pp);
                        // hi = P with its low 13 mantissa bits cleared, lo = the rest (split_pair)
                        const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFFE000u);
                        const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFFE000u);
                        ph[q] = f32x2_to_f16x2(h0, h1);
                        const float2 r = f2_unpack(f2_sub(pp, f2_pack(h0, h1)));
                        pl[q] = f32x2_to_f16x2(r.x, r.y);
                    }
                    tc::st16(s_tm + 32 * c, ph);
                    tc::st16(s_tm + 32 * c + 16, pl);
                }
                const float2 s0 = f2_unpack(ls[0]), s1 = f2_unpack(ls[1]), s2 = f2_unpack(ls[2]), s3 = f2_unpack(ls[3]);
                return ((s0.x + s0.y) + (s1.x + s1.y)) + ((s2.x + s2.y) + (s3.x + s3.y));
            };
            // Publish this half's maximum to the other half's warp (same lane
            // quarter).  While it is in flight, compute P with the running
            // maximum: that is the final P unless a row's maximum grows by more
            // than 2^8 in this tile (then both warps redo it with the new one).
            red_max[(fb * 2 + half) * kRows + row] = mh;
            mbar_arrive(bar(PS::MX + fb * 4 + qtr));
            const bool spec = j > 0 && !__any_sync(kAll, mh > m + 8.f);
            float psum = 0.f;
            if (spec)
                psum = emit(m);
            if (!wwait(bar(PS::MX + fb * 4 + qtr), (j >> 1) & 1, abort_flag, a.err, lane)) {
                ok = false;
                break;
            }
            const float mloc = fmaxf(mh, red_max[(fb * 2 + (half ^ 1)) * kRows + row]);
            bool redo = !spec;
            if (j == 0) {
                m = mloc;                                  // key 0 is visible to every row
            } else {
                // Every kFold tiles the segment accumulator (O_seg, TMEM columns
                // kColO..) is added into O (kColM..) in fp32 and PV_j starts a new
                // segment: the tensor cores' accumulation rounds toward zero, and
                // a chain of thousands of accumulating MMAs (a 128K context is
                // 16K of them) would bias O by ~1e-3 relative.
                const bool fold = (j % kFold) == 0;
                const bool have_o = j > kFold;             // O holds earlier segments
                const bool need = mloc > m + 8.f;
                const bool rescale = __any_sync(kAll, need);
                if (fold || rescale) {
                    // O_seg holds the segment up to tile j-1: wait for that PV.
                    if (!wwait(bar(PS::PV_DONE), (j - 1) & 1, abort_flag, a.err, lane)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const float mn = need ? mloc : m;
                    const float f = rescale ? ex2_approx(m - mn) : 1.f;
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t cs = lanes + kColO + 64 * half + 16 * c;
                        const uint32_t cm = lanes + kColM + 64 * half + 16 * c;
                        uint32_t o[16], t[16];
                        tc::ld16(cs, o);
                        if (have_o)
                            tc::ld16(cm, t);
                        tc::wait_ld();
                        if (fold) {                        // O = (O + O_seg) f
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                t[k] = __float_as_uint(((have_o ? __uint_as_float(t[k]) : 0.f) + __uint_as_float(o[k])) * f);
                            tc::st16(cm, t);
                        } else {                           // both in units of the old maximum
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
                            tc::st16(cs, o);
                            if (have_o) {
#pragma unroll
                                for (int k = 0; k < 16; ++k)
                                    t[k] = __float_as_uint(__uint_as_float(t[k]) * f);
                                tc::st16(cm, t);
                            }
                        }
                    }
                    tc::wait_st();
                    if (rescale) {
                        l *= f;
                        m = mn;
                        redo = true;
                    }
                }
            }
            if (redo)
                psum = emit(m);
            l += psum;
            tc::wait_st();
            tc::fence_before();
            mbar_arrive(bar(PS::P_FULL + fb));
        }
        if (ok && wwait(bar(PS::O_FINAL), 0, abort_flag, a.err, lane)) {
            tc::fence_after();
            red_l[half * kRows + row] = l;
            mbar_arrive(bar(PS::LX + qtr));
            ok = wwait(bar(PS::LX + qtr), 0, abort_flag, a.err, lane);
        } else {
            ok = false;
        }
        if (ok) {
            const float inv = __ldg(a.v_scale + h) / (l + red_l[(half ^ 1) * kRows + row]);
            const int64_t orow = (static_cast<int64_t>(q0) + t0 + tl) * a.hq + h * G + g;
            const bool have_o = nt > kFold;                // at least one segment was folded into O
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[16], t[16];
                tc::ld16(lanes + kColO + 64 * half + 16 * c, o);
                if (have_o)
                    tc::ld16(lanes + kColM + 64 * half + 16 * c, t);
                tc::wait_ld();
                if (!valid)
                    continue;
                float v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    v[k] = ((have_o ? __uint_as_float(t[k]) : 0.f) + __uint_as_float(o[k])) * inv;
                const int d0 = 64 * half + 16 * c;
                if (a.out_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + orow * kHeadDim + d0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + orow * kHeadDim + d0);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * k + 2 * e], v[8 * k + 2 * e + 1]);
                            w[e] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                        dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tm, 512);
    }
}

std::mutex g_prefill_mu;
unsigned long long g_prefill_attr_ctx[64] = {0};   // per device: the context the kernel's limit was raised in

}  // namespace

size_t prefill_smem_bytes()
{
    return PS::bytes();
}

cudaError_t launch_paged_prefill(const PrefillArgs &a, const CUtensorMap &tm_q, const CUtensorMap &tm_k16,
                                 const CUtensorMap &tm_v16, cudaStream_t stream)
{
    const int64_t grid = static_cast<int64_t>(a.batch) * a.hkv * a.max_tiles;
    if (grid <= 0)
        return cudaSuccess;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    {
        unsigned long long ctx = 0;
        const bool known = current_context_id(&ctx);
        std::lock_guard<std::mutex> lk(g_prefill_mu);
        if (!known || g_prefill_attr_ctx[dev] != ctx) {
            e = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(PS::bytes()));
            if (e != cudaSuccess)
                return e;
            g_prefill_attr_ctx[dev] = known ? ctx : 0;
        }
    }
    const int64_t pieces = a.rows_cap * 8;
    int64_t wblocks = (pieces + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (wblocks > cap)
        wblocks = cap;
    if (wblocks < 1)
        wblocks = 1;                                     // CTA 0 always lays out the regions
    const size_t wsmem = (static_cast<size_t>(a.batch) + 1 + 8) * sizeof(int);
    if (wsmem > 48 * 1024) {
        e = cudaFuncSetAttribute(kv_widen_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(wsmem));
        if (e != cudaSuccess)
            return e;
    }
    kv_widen_kernel<<<static_cast<unsigned>(wblocks), 256, wsmem, stream>>>(a);
    paged_prefill_kernel<<<static_cast<unsigned>(grid), kPThreads, PS::bytes(), stream>>>(tm_q, tm_k16, tm_v16, a);
    return cudaGetLastError();
}

}  // namespace pkv
