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
// Design.  One CTA per (sequence, kv head, tile of 128 / G query tokens).  The
// tile's 128 rows are (token, query head of the group) pairs, so each K/V tile
// brought on chip serves all G heads.  Keys are visited in tiles of 128.  One
// role per warp:
//   warp 0      TMA of the bf16 query tile (once, into V buffer 1 for staging);
//   warp 1      owns the 512 TMEM columns and issues tcgen05.mma (one thread):
//                 S_j  = Q K_j^T  M 128 rows, N 128 keys, K 128 dims; A = Q held
//                                 in TMEM, S in TMEM (2 buffers, so S_{j+1}
//                                 overlaps softmax j)
//                 O   += P_j V_j  A = P_j read from TMEM (f16 hi + lo parts),
//                                 B = V_j stored N(=dim)-major
//   warps 2-5   warps 2-3 build K tiles, warps 4-5 V tiles, 64 keys of every
//               tile each.  A warp issues its own TMA copies of its 16-token
//               page pieces into its own 3-stage FP8 ring (block-table entries
//               fetched a tile ahead), then widens E4M3 -> f16 (exact) into the
//               128B-swizzled operand tiles (one K buffer: the QK^T MMAs free
//               it while the previous PV runs; two V buffers).
//               Copies are issued by four warps because each issue costs the
//               issuing thread about as long as a 2 KB copy takes to stream;
//               K and V have their own warps so that K tiles, which the short
//               QK^T MMAs release early, never wait behind V tiles.  These warps
//               also widen the query rows into TMEM at the start;
//   warps 6-13  online softmax, two warps per TMEM lane quarter: one row per
//               thread, each warp one half (64 keys) of the tile.  The row
//               maximum is exchanged through shared memory; exp2 domain, lazy
//               rescaling of O (only when the maximum grows by more than 2^8);
//               P is written over S in TMEM; at the end each warp stores its
//               half of O / l x v_scale.
// Every wait is bounded (2 s): on expiry the CTA sets PKV_DEVERR_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and exits.
#include <mutex>

#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;                       // M: rows of a query tile
constexpr int kKeys = 128;                       // keys per tile
constexpr int kConvWarps = 4;                    // warps 2 .. 5: two for K, two for V
constexpr int kStages = 3;                       // FP8 ring depth of a widening warp
constexpr int kSmWarp0 = 2 + kConvWarps;         // first softmax warp
constexpr int kSmWarps = 8;
constexpr int kPThreads = 32 * (kSmWarp0 + kSmWarps);
constexpr uint32_t kColO = 256, kColQ = 384;     // TMEM columns: S/P 0-255, O 256-383, Q 384-447
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr unsigned kAll = 0xffffffffu;

// Shared memory, offsets from a 1024-byte aligned base.  Operand tiles are
// [2 column blocks][128 rows][128 bytes] with the 128-byte swizzle.
struct PS {
    static constexpr int kTile = 32768;
    static constexpr int kK16 = 0;                    // 1 buffer
    static constexpr int kV16 = kK16 + kTile;         // 2 buffers; buffer 1 first stages the bf16 query tile
    static constexpr int kRing = 4 * 2048;            // one stage of one widening warp: 4 page pieces
    static constexpr int kF8 = kV16 + 2 * kTile;      // [4 warps][kStages][4 pieces][16 rows][128 B]
    static constexpr int kRedMax = kF8 + kConvWarps * kStages * kRing;   // float [2 parities][2 halves][128]
    static constexpr int kRedL = kRedMax + 2048;      // float [2 halves][128 rows]
    static constexpr int kBars = kRedL + 1024;
    enum {
        Q_FULL, Q_READY, K16_FULL, K16_EMPTY, V16_FULL, V16_EMPTY = V16_FULL + 2,
        S_FULL = V16_EMPTY + 2, P_FULL = S_FULL + 2, PV_DONE = P_FULL + 2, O_FINAL, DRAIN,
        MX = DRAIN + 1,                                  // [2 tile parities][4 lane quarters]: row-max exchange
        LX = MX + 8,                                     // [4 lane quarters]: final row-sum exchange
        F8 = LX + 4,                                     // [4 widening warps][kStages]: FP8 pieces landed
        kNumBars = F8 + kConvWarps * kStages
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

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// K-major B operand (128 keys x 128 dims, 128B swizzle), K step s of 16 dims.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int s)
{
    return tc::smem_desc_sw128(tile + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
}

// V as the B operand of O += P V: rows = keys (the K dimension), 128 dims (N)
// contiguous in two 64-dim column blocks 16 KB apart; K step s = keys 16s..16s+15.
__device__ __forceinline__ uint64_t vmn_desc(uint32_t tile, int s)
{
    return tc::smem_desc_sw128(tile + s * 2048, 16384, 1024);
}

// The pieces (16 FP8 bytes each) a widening lane converts for 32 keys: piece
// `it` covers dims 16 e .. 16 e + 15 of local key row kr[it].  Each 8-lane
// phase takes pieces 0-3 of one row and 4-7 of the next (or the other way
// round), so its eight 16-byte reads of the TMA-swizzled FP8 rows and its
// eight pairs of 16-byte stores into the f16 tile land on eight different bank
// groups.
struct PieceMap {
    int kr[8];
    int e;
};

__device__ __forceinline__ PieceMap piece_map(int lane)
{
    PieceMap pm;
    pm.e = lane & 7;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int c = lane + 32 * it;
        pm.kr[it] = 2 * (c >> 4) + ((pm.e >> 2) ^ ((c >> 3) & 1));
    }
    return pm;
}

// FP8 rows of 32 keys (TMA 128B swizzle, rows ring_row0.. of a ring stage) ->
// f16 operand rows kk0.. (exact).  Keys past `last` or in a piece that was not
// loaded (mask bit of its 16-key piece clear) become zeros.  All eight reads
// are issued before any conversion, and the zeroing is a select, so the eight
// read -> convert -> store chains overlap.
__device__ __forceinline__ void widen32(const uint8_t *ring, uint8_t *tile, const PieceMap &pm, int ring_row0,
                                        int kk0, int key0, int last, uint32_t mask)
{
    uint4 v[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int rr = ring_row0 + pm.kr[it];
        v[it] = *reinterpret_cast<const uint4 *>(ring + rr * 128 + ((pm.e ^ (rr & 7)) << 4));
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int rr = ring_row0 + pm.kr[it];
        const int kk = kk0 + pm.kr[it];
        const bool keep = ((mask >> (rr >> 4)) & 1u) && key0 + kk <= last;
        uint4 lo, hi;
        e4m3x4_to_f16x4(keep ? v[it].x : 0u, lo.x, lo.y);
        e4m3x4_to_f16x4(keep ? v[it].y : 0u, lo.z, lo.w);
        e4m3x4_to_f16x4(keep ? v[it].z : 0u, hi.x, hi.y);
        e4m3x4_to_f16x4(keep ? v[it].w : 0u, hi.z, hi.w);
        uint8_t *row = tile + (pm.e >> 2) * 16384 + kk * 128;
        const int c0 = (pm.e & 3) * 2;
        *reinterpret_cast<uint4 *>(row + ((c0 ^ (kk & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(row + (((c0 + 1) ^ (kk & 7)) << 4)) = hi;
    }
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    return f32x2_to_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// P = 2^(x - m) as two f16 parts: hi = x with its low 13 mantissa bits cleared
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

__global__ void __launch_bounds__(kPThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a)
{
    // ---------------------------------------------------------------- the tile
    const int bh_count = a.batch * a.hkv;
    const int rank = blockIdx.x / bh_count;             // heaviest tiles (largest positions) first
    const int bh = blockIdx.x - rank * bh_count;
    const int qt = a.max_tiles - 1 - rank;
    const int b = bh / a.hkv;
    const int h = bh - b * a.hkv;
    const int G = a.group, tpt = a.tokens_per_tile, P = a.page_size;
    const int q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1);
    const int n = q1 - q0;
    const int L = __ldg(a.seq_lens + b);
    if (q0 < 0 || n < 0 || q1 > a.total_q || n > a.max_q_len || L < n ||
        static_cast<int64_t>(L) > static_cast<int64_t>(a.max_pages) * P) {
        if (qt == 0 && h == 0 && threadIdx.x == 0 && a.err)
            atomicOr(a.err, PKV_DEVERR_SEQLEN);
        return;
    }
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
        mbar_init(bar(PS::Q_READY), kConvWarps);
        mbar_init(bar(PS::K16_FULL), kConvWarps / 2);
        mbar_init(bar(PS::K16_EMPTY), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(PS::V16_FULL + i), kConvWarps / 2);
            mbar_init(bar(PS::V16_EMPTY + i), 1);
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
        for (int i = 0; i < kConvWarps * kStages; ++i)
            mbar_init(bar(PS::F8 + i), 1);
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
        // ------------------------------------------------------------ query tile -> staging
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            const uint32_t stage = sb + PS::kV16 + PS::kTile;
            mbar_arrive_expect_tx(bar(PS::Q_FULL), 2u * 128u * G * tpt);
            tma_load_3d(stage, &tm_q, 0, h * G, q0 + t0, bar(PS::Q_FULL), pol);
            tma_load_3d(stage + 16384, &tm_q, 64, h * G, q0 + t0, bar(PS::Q_FULL), pol);
            // The copy must have landed before the CTA may leave.
            pwait(bar(PS::Q_FULL), 0, abort_flag, a.err, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t id_qk = tc::idesc_f16_f32(kRows, kKeys, false);
            const uint32_t id_pv = tc::idesc_f16_f32(kRows, kHeadDim, true);
            const uint32_t o_tm = tm + kColO;
            bool ok = pwait(bar(PS::Q_READY), 0, abort_flag, a.err);
            tc::fence_after();
            for (int j = 0; ok && j <= nt; ++j) {
                if (j < nt) {
                    const int fb = j & 1;
                    if (!pwait(bar(PS::K16_FULL), j & 1, abort_flag, a.err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t kb = sb + PS::kK16;
#pragma unroll
                    for (int s = 0; s < 8; ++s)         // Q dims 16s..16s+15: TMEM columns kColQ + 8s ..
                        tc::mma_ts(tm + fb * 128, tm + kColQ + 8 * s, kmajor_desc(kb, s), id_qk, s > 0);
                    tc::commit(bar_ptr + PS::S_FULL + fb);
                    tc::commit(bar_ptr + PS::K16_EMPTY);
                }
                if (j > 0) {
                    const int i = j - 1, fb = i & 1;
                    if (!pwait(bar(PS::P_FULL + fb), (i >> 1) & 1, abort_flag, a.err) ||
                        !pwait(bar(PS::V16_FULL + fb), (i >> 1) & 1, abort_flag, a.err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t vb = sb + PS::kV16 + fb * PS::kTile;
                    const uint32_t p_tm = tm + fb * 128;
                    // keys 16s..16s+15: hi parts in columns 32(s/2) + 8(s%2) .. +7, lo 16 further
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_ts(o_tm, p_tm + 32 * (s >> 1) + 8 * (s & 1), vmn_desc(vb, s), id_pv,
                                   (i > 0 || s > 0) ? 1u : 0u);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_ts(o_tm, p_tm + 32 * (s >> 1) + 8 * (s & 1) + 16, vmn_desc(vb, s), id_pv, 1u);
                    tc::commit(bar_ptr + PS::PV_DONE);
                    tc::commit(bar_ptr + PS::V16_EMPTY + fb);
                    if (i == nt - 1)
                        tc::commit(bar_ptr + PS::O_FINAL);
                }
            }
            // Every MMA issued has finished before TMEM is released.
            tc::commit(bar_ptr + PS::DRAIN);
            pwait(bar(PS::DRAIN), 0, abort_flag, a.err, false);
        }
    } else if (warp < kSmWarp0) {
        // ------------------------------------------------------------ pages -> f16 operands
        const int cw = warp - 2;
        const bool is_v = cw >= 2;                       // warps 2-3: K, warps 4-5: V
        const CUtensorMap *tmap = is_v ? &tm_v : &tm_k;
        const int kb0 = 64 * (cw & 1);                   // this warp's keys kb0 .. kb0 + 63 of every tile
        const int nbuf = is_v ? 2 : 1;                   // f16 buffers of this tensor
        const int full_bar = is_v ? PS::V16_FULL : PS::K16_FULL;
        const int empty_bar = is_v ? PS::V16_EMPTY : PS::K16_EMPTY;
        const int tile_off = is_v ? PS::kV16 : PS::kK16;
        const uint32_t ring = sb + PS::kF8 + cw * kStages * PS::kRing;
        const uint8_t *ring_p = smem + PS::kF8 + cw * kStages * PS::kRing;
        const PieceMap pm = piece_map(lane);

        // Lanes 0-3 look up the page of piece `lane` (16 keys) of a tile; -1:
        // nothing to load.  The entry is only checked where it is used (issue),
        // so the lookup's latency overlaps a whole tile of work.
        auto fetch_page = [&](int tile) -> int {
            int pg = -1;
            const int k = tile * kKeys + kb0 + 16 * lane;
            if (lane < 4 && tile < nt && k <= last)
                pg = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + k / P);
            return pg;
        };
        // Issues the copies of a tile's pieces into its ring stage; returns the
        // mask of pieces loaded (warp-uniform).  An entry outside the pool sets
        // PKV_DEVERR_PAGE and its piece reads as zeros.
        auto issue = [&](int tile, int pg) -> uint32_t {
            const int k = tile * kKeys + kb0 + 16 * lane;
            if (lane < 4 && tile < nt && k <= last && (pg < 0 || pg >= a.num_pages)) {
                if (a.err)
                    atomicOr(a.err, PKV_DEVERR_PAGE);
                pg = -1;
            }
            const uint32_t mask = __ballot_sync(kAll, pg >= 0) & 0xFu;
            int pgs[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                pgs[i] = __shfl_sync(kAll, pg, i);
            if (lane == 0) {
                const int st = tile % kStages;
                const uint32_t fb8 = bar(PS::F8 + cw * kStages + st);
                mbar_arrive_expect_tx(fb8, __popc(mask) * 2048u);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if ((mask >> i) & 1u)
                        tma_load_3d_plain(ring + st * PS::kRing + i * 2048, tmap, 0,
                                          (tile * kKeys + kb0 + 16 * i) % P, pgs[i] * a.hkv + h, fb8);
            }
            return mask;
        };

        if (lane == 0)
            prefetch_tensormap(tmap);
        uint32_t masks[kStages] = {0, 0, 0};
        int issued = 0;                                  // tiles whose copies were issued
        int pg_next = fetch_page(0);
        for (; issued < kStages - 1 && issued < nt; ++issued) {
            masks[issued] = issue(issued, pg_next);
            pg_next = fetch_page(issued + 1);
        }

        // The query rows: bf16 (staged by TMA, 128B-swizzled) -> f16 in TMEM
        // columns kColQ.. (two dims per column).  Warp w reaches lanes of quarter
        // w % 4, so warps 2-5 cover the 128 rows.
        bool ok = wwait(bar(PS::Q_FULL), 0, abort_flag, a.err, lane);
        if (ok) {
            const int qrow = (warp & 3) * 32 + lane;
            const uint8_t *stage = smem + PS::kV16 + PS::kTile;
            const bool used = qrow < G * tpt;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {            // dims 64 hb .. 64 hb + 63
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (used)
                        v = *reinterpret_cast<const uint4 *>(stage + hb * 16384 + qrow * 128 + ((c ^ (qrow & 7)) << 4));
                    w[4 * c] = bf16x2_to_f16x2(v.x);
                    w[4 * c + 1] = bf16x2_to_f16x2(v.y);
                    w[4 * c + 2] = bf16x2_to_f16x2(v.z);
                    w[4 * c + 3] = bf16x2_to_f16x2(v.w);
                }
                tc::st32(tm + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kColQ + 32 * hb, w);
            }
            tc::wait_st();
            tc::fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(PS::Q_READY));
        }
        int j = 0;
        for (; ok && j < nt; ++j) {
            const int fb = j % nbuf, use = j / nbuf, st = j % kStages;
            if (issued < nt) {                           // keep kStages - 1 tiles in flight
                masks[issued % kStages] = issue(issued, pg_next);
                ++issued;
                pg_next = fetch_page(issued);
            }
            if (!wwait(bar(PS::F8 + cw * kStages + st), (j / kStages) & 1, abort_flag, a.err, lane))
                break;
            if (j >= nbuf && !wwait(bar(empty_bar + fb), (use - 1) & 1, abort_flag, a.err, lane))
                break;
            // V buffer 1 first held the staged query: all four widening warps
            // must be done with it before it is overwritten
            if (is_v && j == 1 && !wwait(bar(PS::Q_READY), 0, abort_flag, a.err, lane))
                break;
#pragma unroll
            for (int gi = 0; gi < 2; ++gi)
                widen32(ring_p + st * PS::kRing, smem + tile_off + fb * PS::kTile, pm, 32 * gi, kb0 + 32 * gi,
                        j * kKeys, last, masks[st]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(full_bar + fb));
        }
        // No copy may still be landing when the CTA leaves.
        if (lane == 0)
            for (int t = j; t < issued; ++t)
                pwait(bar(PS::F8 + cw * kStages + t % kStages), (t / kStages) & 1, abort_flag, a.err, false);
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
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
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
            // pass 1: maximum of the visible scaled logits of this half (hidden
            // keys become -inf here, so pass 2 needs no mask), then of the row
            const int vis = p_row - j * kKeys - 64 * half;
            float mx[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mx[k] = -INFINITY;
            if (vis >= 63) {
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float v = __uint_as_float(x[c][k]) * sl2;
                        x[c][k] = __float_as_uint(v);
                        mx[k & 7] = fmaxf(mx[k & 7], v);
                    }
            } else {
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float v = 32 * c + k <= vis ? __uint_as_float(x[c][k]) * sl2 : -INFINITY;
                        x[c][k] = __float_as_uint(v);
                        mx[k & 7] = fmaxf(mx[k & 7], v);
                    }
            }
            const float mh = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            // exchange with the other half's warp (same lane quarter)
            red_max[(fb * 2 + half) * kRows + row] = mh;
            mbar_arrive(bar(PS::MX + fb * 4 + qtr));
            if (!wwait(bar(PS::MX + fb * 4 + qtr), (j >> 1) & 1, abort_flag, a.err, lane)) {
                ok = false;
                break;
            }
            const float mloc = fmaxf(mh, red_max[(fb * 2 + (half ^ 1)) * kRows + row]);
            if (j == 0) {
                m = mloc;                                  // key 0 is visible to every row
            } else {
                const bool need = mloc > m + 8.f;
                if (__any_sync(kAll, need)) {
                    // O holds the sum up to tile j-1: wait for that PV, then rescale this half of O.
                    if (!wwait(bar(PS::PV_DONE), (j - 1) & 1, abort_flag, a.err, lane)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const float mn = need ? mloc : m;
                    const float f = ex2_approx(m - mn);
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t o[32];
                        tc::ld32(lanes + kColO + 64 * half + 32 * c, o);
                        tc::wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
                        tc::st32(lanes + kColO + 64 * half + 32 * c, o);
                    }
                    tc::wait_st();
                    l *= f;
                    m = mn;
                }
            }
            // pass 2: P = 2^(x - m) <= 2^8 as f16 hi + lo, written over each
            // 32-column piece of S (hi in its first 16 columns, lo in the last 16)
            float ls[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                ls[k] = 0.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t ph[16], pl[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float p0 = ex2_approx(__uint_as_float(x[c][2 * q]) - m);
                    const float p1 = ex2_approx(__uint_as_float(x[c][2 * q + 1]) - m);
                    ls[(2 * q) & 7] += p0;
                    ls[(2 * q + 1) & 7] += p1;
                    split_pair(p0, p1, ph[q], pl[q]);
                }
                tc::st16(s_tm + 32 * c, ph);
                tc::st16(s_tm + 32 * c + 16, pl);
            }
            l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
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
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t o[32];
                tc::ld32(lanes + kColO + 64 * half + 32 * c, o);
                tc::wait_ld();
                if (!valid)
                    continue;
                const int d0 = 64 * half + 32 * c;
                if (a.out_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + orow * kHeadDim + d0);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                             __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + orow * kHeadDim + d0);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(o[8 * k + 2 * e]) * inv,
                                                                     __uint_as_float(o[8 * k + 2 * e + 1]) * inv);
                            w[e] = *reinterpret_cast<uint32_t *>(&v);
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
bool g_prefill_attr[64] = {false};

}  // namespace

size_t prefill_smem_bytes()
{
    return PS::bytes();
}

cudaError_t launch_paged_prefill(const PrefillArgs &a, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                 const CUtensorMap &tm_v, cudaStream_t stream)
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
        std::lock_guard<std::mutex> lk(g_prefill_mu);
        if (!g_prefill_attr[dev]) {
            e = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(PS::bytes()));
            if (e != cudaSuccess)
                return e;
            g_prefill_attr[dev] = true;
        }
    }
    paged_prefill_kernel<<<static_cast<unsigned>(grid), kPThreads, PS::bytes(), stream>>>(tm_q, tm_k, tm_v, a);
    return cudaGetLastError();
}

}  // namespace pkv
