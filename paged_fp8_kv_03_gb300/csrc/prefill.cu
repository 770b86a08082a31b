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
// brought on chip serves all G heads.  Eight warps, one role each:
//   warp 0     TMA: the bf16 query tile once, then per 128-key tile eight
//              16-token FP8 boxes of K and of V, addressed through the block
//              table, into a 2-stage ring;
//   warp 1     owns 512 TMEM columns and issues tcgen05.mma (one thread):
//                S_j  = Q K_j^T  M 128 rows, N 128 keys, K 128 dims -> TMEM
//                                (2 buffers, so S_{j+1} overlaps softmax j)
//                O   += P_j V_j  A = P_j read from TMEM (f16 hi + lo parts),
//                                B = V_j stored N(=dim)-major
//   warps 2-3  widen FP8 -> f16 (exact) into 128B-swizzled operand tiles
//              (2 buffers each for K and V); widen the query tile once;
//   warps 4-7  one thread per row (= TMEM lane): online softmax in the exp2
//              domain with lazy rescaling of O (only when the running maximum
//              grows by more than 2^8), P written over S in TMEM, and at the
//              end O / l x v_scale stored as the output row.
// Every wait is bounded (2 s): on expiry the CTA sets PKV_DEVERR_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and exits.
#include <mutex>

#include "internal.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;                   // M: rows of a query tile
constexpr int kKeys = 128;                   // keys per tile
constexpr int kPThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr unsigned kAll = 0xffffffffu;

// Shared memory, offsets from a 1024-byte aligned base.  Operand tiles are
// [2 column blocks][128 rows][128 bytes] with the 128-byte swizzle.
struct PS {
    static constexpr int kQ = 0;                      // query tile, f16 after widening
    static constexpr int kTile = 32768;
    static constexpr int kK16 = kQ + kTile;           // 2 buffers
    static constexpr int kV16 = kK16 + 2 * kTile;     // 2 buffers
    static constexpr int kF8 = kV16 + 2 * kTile;      // 2 stages x (K 16 KB, V 16 KB)
    static constexpr int kBars = kF8 + 2 * kTile;
    enum {
        Q_FULL, Q_READY, F8_FULL, F8_EMPTY = F8_FULL + 2, K16_FULL = F8_EMPTY + 2, K16_EMPTY = K16_FULL + 2,
        V16_FULL = K16_EMPTY + 2, V16_EMPTY = V16_FULL + 2, S_FULL = V16_EMPTY + 2, P_FULL = S_FULL + 2,
        PV_DONE = P_FULL + 2, O_FINAL, DRAIN, kNumBars
    };
    static constexpr int kMask = kBars + kNumBars * 8;   // chunk masks of the 2 stages
    static constexpr int kTmem = kMask + 8;
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

// K-major operand (rows x 128 dims, 128B swizzle), K step s of 16 dims.
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

// FP8 tile (rows of 128 bytes, TMA 128B swizzle) -> f16 operand tile; rows
// whose chunk was not loaded (mask bit clear) or whose key lies past `last`
// become zeros.  64 threads, 16 B of FP8 -> 32 B of f16 per step.
__device__ __forceinline__ void widen_tile(const uint8_t *src, uint8_t *dst, uint32_t mask, int key0, int last,
                                           int ctid)
{
#pragma unroll 4
    for (int it = 0; it < 16; ++it) {
        const int c = ctid + 64 * it;
        const int kk = c >> 3, dc = c & 7;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
        if (((mask >> (kk >> 4)) & 1u) && key0 + kk <= last) {
            const uint4 v = *reinterpret_cast<const uint4 *>(src + kk * 128 + ((dc ^ (kk & 7)) << 4));
            e4m3x4_to_f16x4(v.x, lo.x, lo.y);
            e4m3x4_to_f16x4(v.y, lo.z, lo.w);
            e4m3x4_to_f16x4(v.z, hi.x, hi.y);
            e4m3x4_to_f16x4(v.w, hi.z, hi.w);
        }
        uint8_t *row = dst + (dc >> 2) * 16384 + kk * 128;
        const int c0 = (dc & 3) * 2;
        *reinterpret_cast<uint4 *>(row + ((c0 ^ (kk & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(row + (((c0 + 1) ^ (kk & 7)) << 4)) = hi;
    }
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    return f32x2_to_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
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
    uint32_t *masks = reinterpret_cast<uint32_t *>(smem + PS::kMask);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + PS::kTmem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + PS::kFlag);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(PS::Q_FULL), 1);
        mbar_init(bar(PS::Q_READY), 2);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(PS::F8_FULL + i), 1);
            mbar_init(bar(PS::F8_EMPTY + i), 2);
            mbar_init(bar(PS::K16_FULL + i), 2);
            mbar_init(bar(PS::K16_EMPTY + i), 1);
            mbar_init(bar(PS::V16_FULL + i), 2);
            mbar_init(bar(PS::V16_EMPTY + i), 1);
            mbar_init(bar(PS::S_FULL + i), 1);
            mbar_init(bar(PS::P_FULL + i), 128);
        }
        mbar_init(bar(PS::PV_DONE), 1);
        mbar_init(bar(PS::O_FINAL), 1);
        mbar_init(bar(PS::DRAIN), 1);
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
    const uint32_t tm = *tslot;           // columns: S/P buffer 0 | S/P buffer 1 | O | unused

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_last();
            mbar_arrive_expect_tx(bar(PS::Q_FULL), 2u * 128u * G * tpt);
            tma_load_3d(sb + PS::kQ, &tm_q, 0, h * G, q0 + t0, bar(PS::Q_FULL), pol);
            tma_load_3d(sb + PS::kQ + 16384, &tm_q, 64, h * G, q0 + t0, bar(PS::Q_FULL), pol);
            uint32_t armed[2] = {0, 0};
            for (int j = 0; j < nt; ++j) {
                const int st = j & 1;
                if (j >= 2 && !pwait(bar(PS::F8_EMPTY + st), ((j >> 1) - 1) & 1, abort_flag, a.err))
                    break;
                const int key0 = j * kKeys;
                int phys[8];
                uint32_t mask = 0, cnt = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    phys[i] = -1;
                    const int k = key0 + 16 * i;
                    if (k > last)
                        continue;
                    const int pg = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + k / P);
                    if (pg < 0 || pg >= a.num_pages) {
                        if (a.err)
                            atomicOr(a.err, PKV_DEVERR_PAGE);
                        continue;
                    }
                    phys[i] = pg;
                    mask |= 1u << i;
                    ++cnt;
                }
                masks[st] = mask;
                mbar_arrive_expect_tx(bar(PS::F8_FULL + st), cnt * 4096u);
                armed[st] = static_cast<uint32_t>(j >> 1) + 1;
                const uint32_t dst = sb + PS::kF8 + st * PS::kTile;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (phys[i] < 0)
                        continue;
                    const int y = (key0 + 16 * i) % P;
                    const int z = phys[i] * a.hkv + h;
                    tma_load_3d(dst + i * 2048, &tm_k, 0, y, z, bar(PS::F8_FULL + st), pol);
                    tma_load_3d(dst + 16384 + i * 2048, &tm_v, 0, y, z, bar(PS::F8_FULL + st), pol);
                }
            }
            // No copy may still be landing when the CTA leaves.
            for (int st = 0; st < 2; ++st)
                if (armed[st])
                    pwait(bar(PS::F8_FULL + st), (armed[st] - 1) & 1, abort_flag, a.err, false);
            // The query tile was armed unconditionally.
            pwait(bar(PS::Q_FULL), 0, abort_flag, a.err, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t id_qk = tc::idesc_f16_f32(kRows, kKeys, false);
            const uint32_t id_pv = tc::idesc_f16_f32(kRows, kHeadDim, true);
            const uint32_t qa = sb + PS::kQ;
            const uint32_t o_tm = tm + 256;
            bool ok = pwait(bar(PS::Q_READY), 0, abort_flag, a.err);
            tc::fence_after();
            for (int j = 0; ok && j <= nt; ++j) {
                if (j < nt) {
                    const int fb = j & 1;
                    if (!pwait(bar(PS::K16_FULL + fb), (j >> 1) & 1, abort_flag, a.err)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const uint32_t kb = sb + PS::kK16 + fb * PS::kTile;
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_ss(tm + fb * 128, kmajor_desc(qa, s), kmajor_desc(kb, s), id_qk, s > 0);
                    tc::commit(bar_ptr + PS::S_FULL + fb);
                    tc::commit(bar_ptr + PS::K16_EMPTY + fb);
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
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_ts(o_tm, p_tm + s * 8, vmn_desc(vb, s), id_pv, (i > 0 || s > 0) ? 1u : 0u);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_ts(o_tm, p_tm + 64 + s * 8, vmn_desc(vb, s), id_pv, 1u);
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
    } else if (warp < 4) {
        // ------------------------------------------------------------ FP8 -> f16
        const int ctid = threadIdx.x - 64;
        bool ok = wwait(bar(PS::Q_FULL), 0, abort_flag, a.err, lane);
        if (ok) {
            const int rows_used = G * tpt;
            for (int i = ctid; i < 2048; i += 64) {          // 16-byte chunks of the query tile
                uint4 *p = reinterpret_cast<uint4 *>(smem + PS::kQ + i * 16);
                const int row = (i >> 3) & 127;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (row < rows_used) {
                    const uint4 w = *p;
                    v = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z),
                                   bf16x2_to_f16x2(w.w));
                }
                *p = v;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(PS::Q_READY));
        }
        for (int j = 0; ok && j < nt; ++j) {
            const int st = j & 1, use = j >> 1;
            if (!wwait(bar(PS::F8_FULL + st), use & 1, abort_flag, a.err, lane))
                break;
            const uint32_t mask = masks[st];
            const int key0 = j * kKeys;
            const uint8_t *f8 = smem + PS::kF8 + st * PS::kTile;
            if (j >= 2 && !wwait(bar(PS::K16_EMPTY + st), (use - 1) & 1, abort_flag, a.err, lane))
                break;
            widen_tile(f8, smem + PS::kK16 + st * PS::kTile, mask, key0, last, ctid);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(PS::K16_FULL + st));
            if (j >= 2 && !wwait(bar(PS::V16_EMPTY + st), (use - 1) & 1, abort_flag, a.err, lane))
                break;
            widen_tile(f8 + 16384, smem + PS::kV16 + st * PS::kTile, mask, key0, last, ctid);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(PS::V16_FULL + st));
                mbar_arrive(bar(PS::F8_EMPTY + st));
            }
        }
    } else {
        // ------------------------------------------------------------ softmax + output
        const int sw = warp - 4;                         // TMEM lane quarter of this warp
        const int row = sw * 32 + lane;
        const int tl = row / G;
        const int g = row - tl * G;
        const bool valid = row < G * tpt && tl < nv;
        const int p_row = valid ? pos0 + tl : last;      // padding rows mirror the last row
        const float sl2 = __ldg(a.k_scale + h) * a.sm_scale_log2;
        const uint32_t lanes = tm + (static_cast<uint32_t>(sw * 32) << 16);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            const int fb = j & 1;
            if (!wwait(bar(PS::S_FULL + fb), (j >> 1) & 1, abort_flag, a.err, lane)) {
                ok = false;
                break;
            }
            tc::fence_after();
            uint32_t x[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tc::ld32(lanes + fb * 128 + 32 * c, x[c]);
            tc::wait_ld();
            const int key0 = j * kKeys;
            float mloc = -INFINITY;
            if (key0 + kKeys - 1 <= p_row) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float v = __uint_as_float(x[c][k]) * sl2;
                        x[c][k] = __float_as_uint(v);
                        mloc = fmaxf(mloc, v);
                    }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float v = (key0 + 32 * c + k <= p_row) ? __uint_as_float(x[c][k]) * sl2 : -INFINITY;
                        x[c][k] = __float_as_uint(v);
                        mloc = fmaxf(mloc, v);
                    }
            }
            if (j == 0) {
                m = mloc;                                  // key 0 is visible to every row
            } else {
                const bool need = mloc > m + 8.f;
                if (__any_sync(kAll, need)) {
                    // O holds the sum up to tile j-1: wait for that PV, then rescale.
                    if (!wwait(bar(PS::PV_DONE), (j - 1) & 1, abort_flag, a.err, lane)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const float mn = need ? mloc : m;
                    const float f = ex2_approx(m - mn);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tc::ld32(lanes + 256 + 32 * c, o);
                        tc::wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
                        tc::st32(lanes + 256 + 32 * c, o);
                    }
                    tc::wait_st();
                    l *= f;
                    m = mn;
                }
            }
            // P = 2^(x - m) <= 2^8, as f16 hi + lo (hi + lo = P to about 2^-22
            // relative), written over S: hi in columns 0..63, lo in 64..127.
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t ph[32], pl[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int c = 2 * half + (q >> 4), k = (q & 15) * 2;
                    const float p0 = ex2_approx(__uint_as_float(x[c][k]) - m);
                    const float p1 = ex2_approx(__uint_as_float(x[c][k + 1]) - m);
                    l += p0 + p1;
                    const uint32_t hv = f32x2_to_f16x2(p0, p1);
                    const float2 hf = f16x2_to_f32x2(hv);
                    ph[q] = hv;
                    pl[q] = f32x2_to_f16x2(p0 - hf.x, p1 - hf.y);
                }
                tc::st32(lanes + fb * 128 + 32 * half, ph);
                tc::st32(lanes + fb * 128 + 64 + 32 * half, pl);
            }
            tc::wait_st();
            tc::fence_before();
            mbar_arrive(bar(PS::P_FULL + fb));
        }
        if (ok && wwait(bar(PS::O_FINAL), 0, abort_flag, a.err, lane)) {
            tc::fence_after();
            const float inv = __ldg(a.v_scale + h) / l;
            const int64_t orow = (static_cast<int64_t>(q0) + t0 + tl) * a.hq + h * G + g;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tc::ld32(lanes + 256 + 32 * c, o);
                tc::wait_ld();
                if (!valid)
                    continue;
                if (a.out_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + orow * kHeadDim + 32 * c);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                             __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
                } else {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + orow * kHeadDim +
                                                           32 * c);
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
