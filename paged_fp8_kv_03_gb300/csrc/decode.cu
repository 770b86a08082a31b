// paged_gqa_decode: grouped-query decode attention over the paged FP8 cache.
//
// What it computes (one query per sequence, every cached token):
//   s_t = sm_scale * q . dequant(K_t),  w = softmax(s),  o = sum_t w_t dequant(V_t)
// with 8 KV heads serving 32 or 64 query heads ("FP8量化与长上下文实测：Llama 3
// 70B部署优化指南", §1.2), K/V stored as E4M3 with a per-(layer, kv head) fp32
// scale (same guide §3.2), tokens reached through a block table of 16- or
// 32-token pages (0539edu.com Llama 3 notes §2.2, §5.2; mlqm.cn Llama 3 8B
// notes §3.3 for 32).  Decode re-reads the whole cache every step and is
// bound by memory bandwidth (0539edu.com notes §3.2; guide §3.3), so the
// design streams every KV byte exactly once at full HBM rate.
//
// Work split.  The (sequence, kv head) segments are laid end to end as one
// list of 16-token chunks (one chunk of one kv head, 2 x 16 x 128 bytes), kv head
// by kv head (every sequence's segment of head 0, then of head 1, ...).  Every
// warp of the persistent grid is an independent worker that takes a
// contiguous range of that list, whatever the sequence lengths (split-K /
// flash-decoding): an equal share, or a share proportional to its CTA's
// weight when the host has installed weights for this grid (the CTAs land on
// the same SMs call after call, and some SMs stream slower than others, so
// calibrated weights let every worker finish at the same time); the shares
// count a few empty "ghost" chunks after every segment, the cost of the
// extra piece a range holding a segment's end carries.  A worker's range
// cuts segments into pieces; a piece covering a whole segment writes the
// final output, the others write a partial softmax state (running max m, sum
// l, unnormalised accumulator) into workspace slot worker + (the segment's
// rank in the list).  A second kernel, one warp per (segment, query head),
// merges the pieces in worker order (deterministic); it is a programmatic
// dependent launch, so it is already resident when the first kernel's last
// warps finish.  With the fused append, the worker that consumes the chunk
// holding a new token stores it to the pool and patches its own copy of the
// chunk, so the call never reads its own store back.
//
// Inside a worker (one warp): lane 0 issues two TMA tensor loads per page
// (K tile, V tile; 128-byte swizzled, evict-first in L2) into the warp's own
// 4-stage shared-memory ring (2 stages of 32-token pages), each stage guarded
// by one mbarrier; the warp refills a stage as soon as it has consumed it, so
// no cross-warp handshake sits on the load path.  Block-table entries come in
// 32 at a time, one batch ahead.  The warp reads a 16-token tile with
// ldmatrix (conflict-free thanks to the swizzle), widens E4M3 to f16 exactly
// in registers, and runs both products on the tensor cores with mma.sync
// m16n8k16 (f16 in, f32 accumulate):
//   S[g][t]   = Q[g][:] . K[t][:]    (A = Q, the group's <= 8 heads; B = K)
//   O^T[d][g] += V^T[d][t] P^T[t][g]  (A = V via ldmatrix.trans; B = P)
// The QK^T output fragment is already laid out as the PV B fragment, so the
// probabilities never leave registers.  P is split into f16 hi + lo parts
// (two PV products) so the probabilities keep ~22 significant bits.  The
// online softmax runs in the exp2 domain with a lazy rescale (only when a
// running max grows by more than 2^8).
//
// Every wait on an mbarrier is bounded (2 s on the global timer): on expiry
// the kernel raises PKV_DEVERR_TIMEOUT, stops issuing copies, drains the ones
// in flight and returns.
#include <math.h>

#include <mutex>

#include "internal.h"

namespace pkv {

namespace {

constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr unsigned kFull = 0xffffffffu;

struct Loc {
    int b, h, ck;   // sequence, kv head, 16-token chunk index within the sequence
};

constexpr int kChunk = 16;   // tokens per chunk: one TMA box, one mma tile

__device__ __forceinline__ int clamp_len(int L, int cap)
{
    return L < 0 ? 0 : (L > cap ? cap : L);
}

// log2 of sequence b's page size in tokens (its pages are runs of
// P_b / page_size consecutive pool pages), or -1 if P_b is not a power of two
// in [page_size, 256].
__device__ __forceinline__ int page_log2_of(const DecodeArgs &a, int b)
{
    if (a.page_sizes == nullptr)
        return a.pool_log2;
    const int pb = __ldg(a.page_sizes + b);
    if (pb < a.page_size || pb > 256 || (pb & (pb - 1)) != 0)
        return -1;
    return 31 - __clz(pb);
}

// Tokens of sequence b the call attends: seq_lens[b] clamped to [0, min(max_len,
// max_pages * P_b)]; 0 for an invalid page size.
__device__ __forceinline__ int seq_len_of(const DecodeArgs &a, int b)
{
    const int lp = page_log2_of(a, b);
    if (lp < 0)
        return 0;
    const long long cap_pages = static_cast<long long>(a.max_pages) << lp;
    const int cap = cap_pages < a.max_len ? static_cast<int>(cap_pages) : a.max_len;
    return clamp_len(__ldg(a.seq_lens + b), cap);
}

// Pool page and row of token t of sequence b (lp = page_log2_of): entry
// bt[b][t / P_b] is the first pool page of the run holding the logical page,
// offset o = t % P_b lies in pool page entry + o / P, row o % P.  Returns
// false for an entry outside the pool.
__device__ __forceinline__ bool token_page(const DecodeArgs &a, int b, int lp, int t, int &phys, int &row)
{
    const int entry = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + (t >> lp));
    const int o = t & ((1 << lp) - 1);
    if (entry < 0 || entry >= a.num_pages)
        return false;
    phys = entry + (o >> a.pool_log2);
    row = o & (a.page_size - 1);
    return phys < a.num_pages;
}

__device__ __forceinline__ int chunks_of(const int *ps, int b)
{
    return ps[b + 1] - ps[b];
}

// The list is head-major: all sequences' chunks of kv head 0, then of head 1,
// ...; segment (b, h) covers list positions [h*ps[batch] + ps[b], ... + np_b).
// (Head-major keeps a batch's short sequences apart in the list, so a
// worker's range crosses fewer segment boundaries than with the heads of one
// sequence side by side.)
__device__ Loc locate(const int *ps, int batch, int hkv, int64_t x)
{
    const int64_t per_head = ps[batch];                  // chunks of one head over all sequences
    Loc l;
    l.h = static_cast<int>(x / per_head);
    const int rem = static_cast<int>(x - static_cast<int64_t>(l.h) * per_head);
    int lo = 0, hi = batch - 1;                          // the last sequence starting at or before rem
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ps[mid] <= rem)
            lo = mid;
        else
            hi = mid - 1;
    }
    l.b = lo;
    l.ck = rem - ps[lo];
    (void)hkv;
    return l;
}

// n chunk-heads further along the list (past its end: h == hkv).
__device__ Loc advance(const int *ps, int batch, int hkv, Loc l, int64_t n)
{
    int64_t pg = l.ck + n;
    while (l.h < hkv) {
        const int np = chunks_of(ps, l.b);
        if (pg < np)
            break;
        pg -= np;
        if (++l.b == batch) {
            l.b = 0;
            ++l.h;
        }
    }
    l.ck = static_cast<int>(pg);
    return l;
}

// Weighted split: prefix sums of the per-CTA weights of the current device
// (entry c = sum of the weights of CTAs 0 .. c-1), written by the host between
// calls; and the calibration's per-CTA start / end times (global timer, ns).
__device__ uint32_t g_split_prefix[kMaxSplitCtas + 1];
__device__ unsigned long long g_split_probe[kMaxSplitCtas][2];

// The split of one call.  pre == nullptr: the even split (C(w) = w, CT = workers).
struct Split {
    const uint32_t *pre;   // weight prefix sums (global or shared memory), num_ctas + 1 entries
    int ctas;
    int64_t ct;            // C(workers)
};

__device__ __forceinline__ Split make_split(const DecodeArgs &a, const uint32_t *pre)
{
    Split sp;
    sp.ctas = a.num_ctas;
    sp.pre = a.split ? pre : nullptr;
    sp.ct = a.split ? a.split_ct : static_cast<int64_t>(a.num_ctas) * kWarps;
    return sp;
}

// List position T * cw / CT of weight position cw = C(w), clamped to [0, T],
// so even a table rewritten during a call (a misuse) keeps every range, and
// so every slot index, inside the list.
__device__ __forceinline__ int64_t range_at(const Split &sp, int64_t total, int64_t cw)
{
    const int64_t x = total * cw / sp.ct;
    return x < 0 ? 0 : (x > total ? total : x);
}

// C(j) for warp j in [0, kWarps] of CTA c, given the CTA's prefix sums p0 =
// P(c) and p1 = P(c + 1) (C(4) is C of the next CTA's warp 0); even split: 4c + j.
__device__ __forceinline__ int64_t split_cw(const Split &sp, int c, int j, uint32_t p0, uint32_t p1)
{
    if (sp.pre == nullptr)
        return static_cast<int64_t>(c) * kWarps + j;
    return static_cast<int64_t>(kWarps) * p0 + static_cast<int64_t>(j) * (p1 - p0);
}

// First list position of worker w's range, T * C(w) / CT (w = workers gives T).
__device__ __forceinline__ int64_t range_lo(const Split &sp, int64_t total, int w)
{
    const int c = w / kWarps, j = w % kWarps;
    if (sp.pre == nullptr)
        return range_at(sp, total, split_cw(sp, c, j, 0u, 0u));
    return range_at(sp, total, c >= sp.ctas ? sp.ct : split_cw(sp, c, j, sp.pre[c], sp.pre[c + 1]));
}

// Real list position of virtual position xv in the list with `ghost` empty
// chunks after every segment (ghost = 0: xv itself): in kv head h's part, the
// largest sequence b with ps[b] + ghost * b <= rem holds it, at real offset
// min(rem - ps[b] - ghost * b, its chunks).
__device__ __forceinline__ int64_t real_position(const int *ps, int batch, int hkv, int ghost, int64_t xv)
{
    const int64_t per_head = ps[batch], per_head_v = per_head + static_cast<int64_t>(ghost) * batch;
    if (per_head_v == 0 || xv >= per_head_v * hkv)
        return per_head * hkv;
    const int64_t h = xv / per_head_v, rem = xv - h * per_head_v;
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ps[mid] + static_cast<int64_t>(ghost) * mid <= rem)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int64_t c = rem - ps[lo] - static_cast<int64_t>(ghost) * lo;
    const int np = ps[lo + 1] - ps[lo];
    return h * per_head + ps[lo] + (c < np ? c : np);
}

struct Smem {
    static constexpr int kTile = kChunk * kHeadDim;         // bytes of one K (or V) chunk tile
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kStages = 4;                       // per warp: 16 KB ring
    static constexpr int kWarpRing = kStages * kStageBytes;
    static constexpr int kBar = kWarps * kWarpRing;         // full[kWarps][kStages]
    static constexpr int kFlag = kBar + kWarps * kStages * 8;   // abort flag
    static constexpr int kWarpSum = kFlag + 16;             // scan scratch (kWarps ints)
    static constexpr int kFoldM = kWarpSum + 32;            // per warp: the running maximum of each head at its last fold
    static constexpr int kArgs = kFoldM + kWarps * PKV_MAX_GROUP * 4;   // a copy of the call's arguments
    static constexpr int kPstart = kArgs + (static_cast<int>(sizeof(DecodeArgs)) + 15) / 16 * 16;
    static size_t bytes(int batch) { return static_cast<size_t>(kPstart) + 4u * (batch + 1) + 1024u; }
};

// Bounded wait by a whole warp (all lanes get acquire semantics); warp-uniform.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *err, int lane)
{
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        const bool done = mbar_try_wait(bar, parity);
        if (__all_sync(kFull, done))
            return true;
        if ((it & 15u) == 15u) {
            int stop = 0;
            if (lane == 0) {
                if (*abort_flag) {
                    stop = 1;
                } else if (t0 == 0) {
                    t0 = global_timer_ns();
                } else if (global_timer_ns() - t0 > kTimeoutNs) {
                    *abort_flag = 1;
                    if (err)
                        atomicOr(err, PKV_DEVERR_TIMEOUT);
                    stop = 1;
                }
            }
            if (__shfl_sync(kFull, stop, 0))
                return false;
        }
    }
}

// Bounded wait by a single thread.
__device__ __forceinline__ bool wait_thread(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                            int32_t *err, bool honour_abort)
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
            if (global_timer_ns() - t0 > kTimeoutNs) {
                *abort_flag = 1;
                if (err)
                    atomicOr(err, PKV_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void store_out(const DecodeArgs &a, int64_t row, int d, float v)
{
    if (a.out_f32)
        static_cast<float *>(a.out)[row * kHeadDim + d] = v;
    else
        static_cast<__nv_bfloat16 *>(a.out)[row * kHeadDim + d] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ void store_pair(const DecodeArgs &a, int64_t row, int d, float v0, float v1)
{
    if (a.out_f32)
        *reinterpret_cast<float2 *>(static_cast<float *>(a.out) + row * kHeadDim + d) = make_float2(v0, v1);
    else
        *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(a.out) + row * kHeadDim + d) =
            __floats2bfloat162_rn(v0, v1);
}

// Per-lane byte offsets of the ldmatrix rows inside a 16-token tile (128-byte
// rows, 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7)).
// x4 load q covers: K -> matrices (j, sg) = (mi & 1, 2q + (mi >> 1)), rows
// 8j..8j+7; V -> the same pattern over (token half, dim segment).
struct TileOffsets {
    uint32_t ld[4];
};

__device__ __forceinline__ TileOffsets tile_offsets(int lane)
{
    TileOffsets o;
    const int r = lane & 7, mi = lane >> 3;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int half = mi & 1, sg = 2 * q + (mi >> 1), tok = 8 * half + r;
        o.ld[q] = static_cast<uint32_t>(tok * kHeadDim + ((sg ^ r) << 4));
    }
    return o;
}

// One 16-token tile (already in registers, see load_tile): scores, online
// softmax update, P.V accumulation.  nv: valid tokens in the tile (1..16);
// kPartial when nv < 16.
// Instruction order keeps dependent tensor-core ops apart: QK^T runs as four
// independent accumulator chains, and the two PV products of an accumulator
// are four MMAs apart.
struct TileFrags {
    uint32_t kf[2][8];   // K: [token half j][dim segment]
    uint32_t vf[2][8];   // V (transposed pairs): [token half][dim segment]
};

// Copies one 16-token tile from the ring into registers.
__device__ __forceinline__ void load_tile(uint32_t kt, uint32_t vt, const TileOffsets &off, TileFrags &f)
{
#pragma unroll
    for (int q = 0; q < 4; ++q)
        ldsm_x4(kt + off.ld[q], f.kf[0][2 * q], f.kf[1][2 * q], f.kf[0][2 * q + 1], f.kf[1][2 * q + 1]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        ldsm_x4_trans(vt + off.ld[q], f.vf[0][2 * q], f.vf[1][2 * q], f.vf[0][2 * q + 1], f.vf[1][2 * q + 1]);
}

template <bool kPartial>
__device__ __forceinline__ void process_tile(TileFrags &fr, int nv, const uint32_t (&qa)[8][2], float scale2,
                                             float &m_ref, float &lsum, float (&acc)[8][4], int lane)
{
    const int t4 = lane & 3;
    uint32_t (&kf)[2][8] = fr.kf;
    uint32_t (&vf)[2][8] = fr.vf;

    // S = Q K^T.  Thread (gid, t4) gets S[head gid][tokens 8j + 2t4, 8j + 2t4 + 1];
    // even and odd k-steps accumulate separately and are added at the end.
    float sc[2][2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                sc[j][h][c] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t b0, b1;
            e4m3x4_to_f16x4(kf[j][kk], b0, b1);
            mma_16816(sc[j][kk & 1], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
        }

    float y[4] = {(sc[0][0][0] + sc[0][1][0]) * scale2, (sc[0][0][1] + sc[0][1][1]) * scale2,
                  (sc[1][0][0] + sc[1][1][0]) * scale2, (sc[1][0][1] + sc[1][1][1]) * scale2};
    if (kPartial) {
        if (2 * t4 >= nv) y[0] = -INFINITY;
        if (2 * t4 + 1 >= nv) y[1] = -INFINITY;
        if (8 + 2 * t4 >= nv) y[2] = -INFINITY;
        if (9 + 2 * t4 >= nv) y[3] = -INFINITY;
    }
    // Lazy rescale: the running reference m_ref (shared by the 4 lanes of a
    // head) moves only when some score exceeds it by more than 2^8, so the
    // common path needs no cross-lane max.
    const float lmax = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
    if (__any_sync(kFull, lmax > m_ref + kRescaleThreshold)) {
        float tmax = fmaxf(lmax, __shfl_xor_sync(kFull, lmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 2));
        const float m_new = fmaxf(m_ref, tmax);
        const float alpha = ex2_approx(m_ref - m_new);
        lsum *= alpha;
        m_ref = m_new;
        // The accumulator of this thread belongs to heads 2*t4 and 2*t4+1.
        const float a0 = __shfl_sync(kFull, alpha, 8 * t4);
        const float a1 = __shfl_sync(kFull, alpha, 8 * t4 + 4);
#pragma unroll
        for (int sg = 0; sg < 8; ++sg) {
            acc[sg][0] *= a0;
            acc[sg][1] *= a1;
            acc[sg][2] *= a0;
            acc[sg][3] *= a1;
        }
    }
    const float p0 = ex2_approx(y[0] - m_ref), p1 = ex2_approx(y[1] - m_ref);
    const float p2 = ex2_approx(y[2] - m_ref), p3 = ex2_approx(y[3] - m_ref);
    lsum += (p0 + p1) + (p2 + p3);
    const uint32_t h01 = f32x2_to_f16x2(p0, p1), h23 = f32x2_to_f16x2(p2, p3);
    const float2 b01 = f16x2_to_f32x2(h01), b23 = f16x2_to_f32x2(h23);
    const uint32_t l01 = f32x2_to_f16x2(p0 - b01.x, p1 - b01.y);
    const uint32_t l23 = f32x2_to_f16x2(p2 - b23.x, p3 - b23.y);

    if (kPartial) {   // rows past the sequence end may hold anything (even NaN codes)
        const uint32_t m0 = (2 * t4 < nv ? 0x0000FFFFu : 0u) | (2 * t4 + 1 < nv ? 0xFFFF0000u : 0u);
        const uint32_t m1 = (8 + 2 * t4 < nv ? 0x0000FFFFu : 0u) | (9 + 2 * t4 < nv ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int sg = 0; sg < 8; ++sg) {
            vf[0][sg] &= m0;
            vf[1][sg] &= m1;
        }
    }
    // O^T[d][g] += V^T[d][t] P^T[t][g]; dims of m-tile sg: rows gid -> 16sg+2gid, gid+8 -> 16sg+2gid+1.
#pragma unroll
    for (int g4 = 0; g4 < 8; g4 += 4) {
        uint32_t va[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            e4m3x4_to_f16x4(__byte_perm(vf[0][g4 + i], 0, 0x3120), va[i][0], va[i][1]);
            e4m3x4_to_f16x4(__byte_perm(vf[1][g4 + i], 0, 0x3120), va[i][2], va[i][3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            mma_16816(acc[g4 + i], va[i][0], va[i][1], va[i][2], va[i][3], h01, h23);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            mma_16816(acc[g4 + i], va[i][0], va[i][1], va[i][2], va[i][3], l01, l23);
    }
}

// Fused append, one chunk: the worker that consumes chunk ck of segment (b, h)
// (exactly one worker owns each chunk) quantises the step's new tokens that
// fall in it, stores them to the pool for later calls, and writes the same
// bytes into the chunk's copy in its ring, which the TMA filled before (or
// while) the stores reached the pool.  So this call never reads its own
// stores back: no proxy fence, and neither the stores nor the loads wait for
// the other.  Lanes split the 128 dims, 4 each; lane i's 4 bytes of row r sit
// in 16-byte unit (i / 4) XOR (r mod 8) of the row (the TMA's 128-byte swizzle).
// Called after the chunk's wait, before its rows are read.
__device__ __noinline__ void store_new_tokens(const DecodeArgs &a, int b, int h, int ck, int L, uint32_t kt,
                                              uint32_t vt, int lane)
{
    const int lp = page_log2_of(a, b);
    const int t0 = max(ck * kChunk, L - a.n_new), t1 = min(ck * kChunk + kChunk, L);
    for (int t = t0; t < t1; ++t) {
        int phys, row;
        if (!token_page(a, b, lp, t, phys, row))
            continue;   // the chunk's page is outside the pool: flagged at its issue, read as zeros
        const int j = t - (L - a.n_new);
        const int64_t src = ((static_cast<int64_t>(b) * a.n_new + j) * a.hkv + h) * kHeadDim + 4 * lane;
        const int64_t dst = ((static_cast<int64_t>(phys) * a.hkv + h) * a.page_size + row) * kHeadDim + 4 * lane;
        float k4[4], v4[4];
        if (a.new_bf16) {
            const uint2 kb = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(a.k_new) + src));
            const uint2 vb = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(a.v_new) + src));
            k4[0] = __uint_as_float(kb.x << 16); k4[1] = __uint_as_float(kb.x & 0xFFFF0000u);
            k4[2] = __uint_as_float(kb.y << 16); k4[3] = __uint_as_float(kb.y & 0xFFFF0000u);
            v4[0] = __uint_as_float(vb.x << 16); v4[1] = __uint_as_float(vb.x & 0xFFFF0000u);
            v4[2] = __uint_as_float(vb.y << 16); v4[3] = __uint_as_float(vb.y & 0xFFFF0000u);
        } else {
            const float4 kf = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(a.k_new) + src));
            const float4 vf = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(a.v_new) + src));
            k4[0] = kf.x; k4[1] = kf.y; k4[2] = kf.z; k4[3] = kf.w;
            v4[0] = vf.x; v4[1] = vf.y; v4[2] = vf.z; v4[3] = vf.w;
        }
        const uint32_t kq = quantise4(k4[0], k4[1], k4[2], k4[3], __ldg(a.k_scale + h));
        const uint32_t vq = quantise4(v4[0], v4[1], v4[2], v4[3], __ldg(a.v_scale + h));
        *reinterpret_cast<uint32_t *>(a.k_pool + dst) = kq;
        *reinterpret_cast<uint32_t *>(a.v_pool + dst) = vq;
        const int r = t - ck * kChunk;
        const uint32_t off = static_cast<uint32_t>(r * kHeadDim + (((lane >> 2) ^ (r & 7)) << 4) + 4 * (lane & 3));
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(kt + off), "r"(kq) : "memory");
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(vt + off), "r"(vq) : "memory");
    }
    __syncwarp();   // every lane's patch before any lane reads the rows
}

// Segment records for the merge kernel, for the segments this worker's range
// [lo, hi) touches: the worker holding a segment's first chunk writes where
// the segment lies and whether its pieces need merging (-1: its piece is the
// whole segment, the output is final), the worker holding its last chunk
// writes its own index.  Pieces end at a segment's end or the range's end,
// as in the streaming loop.
__device__ __noinline__ void write_records(const DecodeArgs &a, const int *pstart, int64_t lo, int64_t hi, int worker)
{
    Loc l = locate(pstart, a.batch, a.hkv, lo);
    int64_t k = 0;
    const int64_t n_total = hi - lo;
    while (k < n_total && l.h < a.hkv) {
        const int np = chunks_of(pstart, l.b);
        const int n_piece = static_cast<int>(min(static_cast<int64_t>(np - l.ck), n_total - k));
        SegRecord *rec = a.segs + l.b * a.hkv + l.h;
        if (l.ck == 0) {
            rec->start = static_cast<long long>(l.h) * pstart[a.batch] + pstart[l.b];
            rec->n = np;
            rec->w0 = n_piece == np ? -1 : worker;
        }
        if (l.ck + n_piece == np)
            rec->w1 = worker;
        k += n_piece;
        l = advance(pstart, a.batch, a.hkv, l, n_piece);
    }
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    paged_gqa_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const DecodeArgs a)
{
    using S = Smem;
    constexpr int kStages = S::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (a.probe && tid == 0)
        g_split_probe[blockIdx.x][0] = global_timer_ns();
    // This CTA's weight prefix sums P(c), P(c + 1): loaded first, so that the
    // load overlaps the page-offset pass (the ranges need both).
    uint32_t pre_c0 = 0u, pre_c1 = 0u;
    if (a.split) {
        pre_c0 = g_split_prefix[blockIdx.x];
        pre_c1 = g_split_prefix[blockIdx.x + 1];
    }
    int *pstart = reinterpret_cast<int *>(smem + S::kPstart);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kFlag);
    int *warp_sum = reinterpret_cast<int *>(smem + S::kWarpSum);

    // ---- per-sequence page offsets (every CTA computes them; B ints from L2)
    {
        const int chunk = (a.batch + kThreads - 1) / kThreads;
        const int b0 = min(a.batch, tid * chunk), b1 = min(a.batch, b0 + chunk);
        int local = 0;
        for (int b = b0; b < b1; ++b)
            local += (seq_len_of(a, b) + kChunk - 1) / kChunk;
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o)
                incl += v;
        }
        if (lane == 31)
            warp_sum[warp] = incl;
        if (tid == 0) {
            // The out-of-line helpers below take the arguments by reference;
            // given the kernel parameter itself they would read every field
            // through its global address, one memory round trip each at the
            // start of the call, so they get this shared-memory copy.
            *reinterpret_cast<DecodeArgs *>(smem + S::kArgs) = a;
            *abort_flag = 0;
            const uint32_t bar0 = smem_addr(smem + S::kBar);
            for (int s = 0; s < kWarps * kStages; ++s)
                mbar_init(bar0 + 8 * s, 1);
            fence_barrier_init();
        }
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w)
            base += warp_sum[w];
        int run = base + incl - local;
        for (int b = b0; b < b1; ++b) {
            const int L = seq_len_of(a, b);
            pstart[b] = run;
            run += (L + kChunk - 1) / kChunk;
            if (blockIdx.x == 0 && a.err) {
                const int raw = __ldg(a.seq_lens + b);
                if (page_log2_of(a, b) < 0)
                    atomicOr(a.err, PKV_DEVERR_PAGESIZE);
                else if (raw != L || (a.k_new != nullptr && L < a.n_new))
                    atomicOr(a.err, PKV_DEVERR_SEQLEN);
            }
        }
        if (tid == kThreads - 1)
            pstart[a.batch] = base + incl;
        __syncthreads();
    }

    // Sequences with no tokens: nobody streams them, so write their zero rows
    // (and a record telling the merge kernel to skip them) here.
    for (int sg = blockIdx.x; sg < a.batch * a.hkv; sg += a.num_ctas) {
        const int b = sg / a.hkv;
        if (chunks_of(pstart, b) == 0) {
            const int64_t row0 = static_cast<int64_t>(b) * a.hq + static_cast<int64_t>(sg % a.hkv) * a.group;
            for (int e = tid; e < a.group * kHeadDim; e += kThreads)
                store_out(a, row0 + (e >> 7), e & (kHeadDim - 1), 0.f);
            if (tid == 0) {
                a.segs[sg].n = 0;
                a.segs[sg].w0 = -1;
            }
        }
    }

    const int worker = blockIdx.x * kWarps + warp;
    const int64_t total = static_cast<int64_t>(pstart[a.batch]) * a.hkv;
    const Split sp = make_split(a, g_split_prefix);
    if (blockIdx.x == 0 && tid == 0) {
        DecodeHeader hd;
        hd.total = total;
        hd.pad = 0;
        *a.header = hd;
    }
    // Let the merge kernel get scheduled now; it waits for this grid to finish.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // The split runs over a virtual list with kGhostChunks empty chunks after
    // every segment, so that a range holding a segment's end (one more piece:
    // a partial state, the next query rows, the new token) gets that much less
    // real work; its real edges are where the virtual ones fall (a ghost maps
    // to the next segment's start).  Only while every range holds a chunk
    // (T * wmin >= CT): otherwise the plain split, which the merge can walk.
    const int ghost = total * (a.split ? a.split_wmin : 1) >= sp.ct ? kGhostChunks : 0;
    // lane 0 works out the range's start, lane 1 its end
    const int64_t edge = real_position(pstart, a.batch, a.hkv, ghost,
                                       range_at(sp, total + static_cast<int64_t>(ghost) * a.batch * a.hkv,
                                                split_cw(sp, blockIdx.x, warp + (lane & 1), pre_c0, pre_c1)));
    const int64_t lo = __shfl_sync(kFull, edge, 0), hi = __shfl_sync(kFull, edge, 1);
    if (lo >= hi) {                              // warp-level: no CTA barrier follows
        if (a.probe && lane == 0)
            atomicMax(&g_split_probe[blockIdx.x][1], static_cast<unsigned long long>(global_timer_ns()));
        return;
    }
    const int n_total = static_cast<int>(hi - lo);

    // (The fused append needs nothing here: the worker owning a chunk with new
    // tokens stores them when it consumes the chunk, see store_new_tokens.)
    const DecodeArgs &a_s = *reinterpret_cast<const DecodeArgs *>(smem + S::kArgs);

    const uint32_t ring = smem_addr(smem) + warp * S::kWarpRing;
    const uint32_t bars = smem_addr(smem + S::kBar) + warp * kStages * 8;
    const uint64_t policy = l2_policy_evict_first();
    const int zoob = static_cast<int>(a.num_pages * a.hkv);   // first out-of-pool tile: reads zeros
    // TMA coordinates of a chunk: tile z = pool page * hkv + head, row y = the
    // chunk's first row within that pool page.
    auto tile_zy = [&](Loc l) -> int2 {
        int phys, row;
        if (!token_page(a, l.b, page_log2_of(a, l.b), l.ck * kChunk, phys, row)) {
            if (a.err)
                atomicOr(a.err, PKV_DEVERR_PAGE);
            return make_int2(zoob, 0);
        }
        return make_int2(phys * a.hkv + l.h, row);
    };

    // ---- block-table batches: zcur holds chunks [32*fb, 32*fb+32), znext the next 32
    Loc cons = locate(pstart, a.batch, a.hkv, lo);
    Loc nbase = advance(pstart, a.batch, a.hkv, cons, 32);
    int2 zcur = lane < n_total ? tile_zy(advance(pstart, a.batch, a.hkv, cons, lane)) : make_int2(0, 0);
    int2 znext = 32 + lane < n_total ? tile_zy(advance(pstart, a.batch, a.hkv, nbase, lane)) : make_int2(0, 0);
    int fb = 0;
    // Warp-uniform bookkeeping of the ring: bit s of `pending` is set while
    // stage s has a copy in flight that nobody has waited for yet, bit s of
    // `pend_par` is the parity of that fill.  Used only to drain after an abort.
    uint32_t pending = 0, pend_par = 0;

    auto issue = [&](int f) {                    // warp-uniform; chunk f goes to stage f % kStages
        if (f >= 32 * (fb + 1)) {
            zcur = znext;
            ++fb;
            nbase = advance(pstart, a.batch, a.hkv, nbase, 32);
            znext = 32 * (fb + 1) + lane < n_total ? tile_zy(advance(pstart, a.batch, a.hkv, nbase, lane))
                                                   : make_int2(0, 0);
        }
        const int z = __shfl_sync(kFull, zcur.x, f & 31);
        const int y = __shfl_sync(kFull, zcur.y, f & 31);
        // Test hook: the selected worker never loads its first page, so its
        // first wait must run out (failure-detection test; -1 = off).
        const bool withheld = worker == a.withhold_worker && f == 0;
        const int go = __shfl_sync(kFull, (lane == 0 && !*abort_flag && !withheld) ? 1 : 0, 0);
        if (go) {
            const int s = f % kStages;
            if (lane == 0) {
                const uint32_t dst = ring + s * S::kStageBytes;
                mbar_arrive_expect_tx(bars + 8 * s, 2 * S::kTile);
                tma_load_3d(dst, &tm_k, 0, y, z, bars + 8 * s, policy);
                tma_load_3d(dst + S::kTile, &tm_v, 0, y, z, bars + 8 * s, policy);
            }
            pending |= 1u << s;
            pend_par = (pend_par & ~(1u << s)) | ((static_cast<uint32_t>(f / kStages) & 1u) << s);
        }
    };
    for (int f = 0; f < kStages && f < n_total; ++f)
        issue(f);
    // Records: only a range holding some segment's first or last chunk writes one.
    if (cons.ck == 0 || n_total > chunks_of(pstart, cons.b) - cons.ck - 1) {
        if (lane == 0)                           // while the first loads are in flight
            write_records(a_s, pstart, lo, hi, worker);
        __syncwarp();
    }

    const int gid = lane >> 2, t4 = lane & 3;
    const TileOffsets off = tile_offsets(lane);
    int st = 0;                                  // stage of page k
    uint32_t ph = 0;                             // its fill parity
    int k = 0;
    while (k < n_total) {
        const int np = chunks_of(pstart, cons.b);
        // a piece ends at its segment's end or the worker's range end
        const int n_piece = min(np - cons.ck, n_total - k);
        const int slot_index = worker;
        const int L = seq_len_of(a, cons.b);
        const bool whole = (cons.ck == 0) && (n_piece == np);
        // the segment's rank in list order: slot worker + rank is distinct for
        // every piece because worker and rank both grow along the list
        const int rank = cons.h * a.batch + cons.b;
        const float scale2 = __ldg(a.k_scale + cons.h) * a.sm_scale_log2;

        // Q fragment for k-step kk: head gid, dims 16kk + 4t4 + {0,1} and {2,3}.
        uint32_t qa[8][2];
        {
            const bool valid = gid < a.group;
            const __nv_bfloat16 *qrow =
                a.q + (static_cast<int64_t>(cons.b) * a.hq + cons.h * a.group + (valid ? gid : 0)) * kHeadDim;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint2 v = make_uint2(0u, 0u);
                if (valid)
                    v = __ldg(reinterpret_cast<const uint2 *>(qrow + 16 * kk + 4 * t4));
                qa[kk][0] = f32x2_to_f16x2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u));
                qa[kk][1] = f32x2_to_f16x2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
            }
        }

        float m_ref = -INFINITY, lsum = 0.f;
        float acc[8][4];
        // Fold: add the accumulator stored in the piece's slot (if any), rescaled
        // from the maxima it was stored with to the current ones, into acc; with
        // store, write acc back as the new fold and restart acc from zero.  Keeps
        // every tensor-core accumulation chain within kFoldChunks chunks.
        // folded: the slot already holds a fold (after the first kFoldChunks).
        auto fold = [&](bool folded, bool store) {
            const int64_t sidx = static_cast<int64_t>(slot_index) + rank;
            if (sidx >= a.num_slots) {
                if (a.err && lane == 0)
                    atomicOr(a.err, PKV_DEVERR_INTERNAL);
                return;
            }
            float *slot = a.partials + sidx * a.group * kPartialStride;
            float *fm = reinterpret_cast<float *>(smem + S::kFoldM) + warp * PKV_MAX_GROUP;
            const float m0 = __shfl_sync(kFull, m_ref, 8 * t4), m1 = __shfl_sync(kFull, m_ref, 8 * t4 + 4);
            const bool h0 = 2 * t4 < a.group, h1 = 2 * t4 + 1 < a.group;
            const float f0 = (folded && h0) ? ex2_approx(fm[2 * t4] - m0) : 0.f;
            const float f1 = (folded && h1) ? ex2_approx(fm[2 * t4 + 1] - m1) : 0.f;
#pragma unroll
            for (int sg = 0; sg < 8; ++sg) {
                float2 *p0 = reinterpret_cast<float2 *>(slot + (2 * t4) * kPartialStride + 16 * sg + 2 * gid);
                float2 *p1 = reinterpret_cast<float2 *>(slot + (2 * t4 + 1) * kPartialStride + 16 * sg + 2 * gid);
                if (folded && h0) {
                    const float2 v = *p0;
                    acc[sg][0] = fmaf(v.x, f0, acc[sg][0]);
                    acc[sg][2] = fmaf(v.y, f0, acc[sg][2]);
                }
                if (folded && h1) {
                    const float2 v = *p1;
                    acc[sg][1] = fmaf(v.x, f1, acc[sg][1]);
                    acc[sg][3] = fmaf(v.y, f1, acc[sg][3]);
                }
                if (store) {
                    if (h0)
                        *p0 = make_float2(acc[sg][0], acc[sg][2]);
                    if (h1)
                        *p1 = make_float2(acc[sg][1], acc[sg][3]);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        acc[sg][c] = 0.f;
                }
            }
            if (store) {
                __syncwarp();                    // every lane has read the old maxima
                if (t4 == 0 && gid < a.group)
                    fm[gid] = m_ref;
                __syncwarp();
            }
        };
#pragma unroll
        for (int sg = 0; sg < 8; ++sg)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                acc[sg][c] = 0.f;

        for (int j = 0; j < n_piece; ++j, ++k) {
            const int nv = min(kChunk, L - (cons.ck + j) * kChunk);
            const int s = st;
            const uint32_t par = ph;
            if (++st == kStages) {
                st = 0;
                ph ^= 1u;
            }
            const bool ready = wait_warp(bars + 8 * s, par, abort_flag, a.err, lane);
            if (ready)
                pending &= ~(1u << s);
            const uint32_t kt = ring + s * S::kStageBytes;
            if (a.k_new != nullptr && ready && (cons.ck + j + 1) * kChunk > L - a.n_new)
                store_new_tokens(a_s, cons.b, cons.h, cons.ck + j, L, kt, kt + S::kTile, lane);
            // Copy the chunk into registers, then hand the stage straight back
            // to the TMA unit so every stage stays in flight during the math.
            TileFrags fr;
            if (ready)
                load_tile(kt, kt + S::kTile, off, fr);
            if (k + kStages < n_total) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                issue(k + kStages);
            }
            if (ready) {
                if (nv >= kChunk)
                    process_tile<false>(fr, kChunk, qa, scale2, m_ref, lsum, acc, lane);
                else
                    process_tile<true>(fr, nv, qa, scale2, m_ref, lsum, acc, lane);
            }
            if (((j + 1) % kFoldChunks) == 0 && j + 1 < n_piece)
                fold(j + 1 > kFoldChunks, true);
        }
        if (n_piece > kFoldChunks)
            fold(true, false);

        // ---- end of piece
        lsum += __shfl_xor_sync(kFull, lsum, 1);
        lsum += __shfl_xor_sync(kFull, lsum, 2);
        const float vsc = __ldg(a.v_scale + cons.h);
        const int64_t row0 = static_cast<int64_t>(cons.b) * a.hq + cons.h * a.group;
        const bool h0 = 2 * t4 < a.group, h1 = 2 * t4 + 1 < a.group;
        if (whole) {
            const float l0 = __shfl_sync(kFull, lsum, 8 * t4), l1 = __shfl_sync(kFull, lsum, 8 * t4 + 4);
            const float s0 = vsc / l0, s1 = vsc / l1;
#pragma unroll
            for (int sg = 0; sg < 8; ++sg) {
                const int d = 16 * sg + 2 * gid;
                if (h0)
                    store_pair(a, row0 + 2 * t4, d, acc[sg][0] * s0, acc[sg][2] * s0);
                if (h1)
                    store_pair(a, row0 + 2 * t4 + 1, d, acc[sg][1] * s1, acc[sg][3] * s1);
            }
        } else if (static_cast<int64_t>(slot_index) + rank >= a.num_slots) {
            if (a.err && lane == 0)
                atomicOr(a.err, PKV_DEVERR_INTERNAL);
        } else {
            float *slot = a.partials + static_cast<int64_t>(slot_index + rank) * a.group * kPartialStride;
#pragma unroll
            for (int sg = 0; sg < 8; ++sg) {
                const int d = 16 * sg + 2 * gid;
                if (h0)
                    *reinterpret_cast<float2 *>(slot + (2 * t4) * kPartialStride + d) = make_float2(acc[sg][0], acc[sg][2]);
                if (h1)
                    *reinterpret_cast<float2 *>(slot + (2 * t4 + 1) * kPartialStride + d) =
                        make_float2(acc[sg][1], acc[sg][3]);
            }
            if (t4 == 0 && gid < a.group) {
                slot[gid * kPartialStride + kHeadDim] = m_ref;
                slot[gid * kPartialStride + kHeadDim + 1] = lsum;
            }
        }
        cons = advance(pstart, a.batch, a.hkv, cons, n_piece);
    }

    // Drain: never leave with a copy still writing this warp's ring (only
    // possible after an abort: normally every issued page was waited for).
    if (pending != 0 && lane == 0) {
        for (int s = 0; s < kStages; ++s)
            if (pending & (1u << s))
                wait_thread(bars + 8 * s, (pend_par >> s) & 1u, abort_flag, a.err, false);
    }
    if (a.probe && lane == 0)
        atomicMax(&g_split_probe[blockIdx.x][1], static_cast<unsigned long long>(global_timer_ns()));
}

// One warp per (segment, query head g of its group), or kSub warps when the
// segments have many pieces (a CTA per (segment, head) then, so that the
// merge's reads spread over the whole GPU); lane j owns dimensions 4j ..
// 4j+3.  The warps merge the partial states the workers covering the segment
// wrote for head g, in list order, and write the output row.  Pieces are taken 16 at a
// time: lane i finds the slot of piece i and loads its (m, l); every lane
// stages its four dimensions of all 16 accumulators in shared memory; then
// one exact rescale folds the batch into the running (M, L, A).  The order is
// fixed, so results are deterministic.
//
// Where a segment's pieces are: with no empty range, piece i was written by
// worker w0 + i and the last one by w1 (the segment's record); otherwise
// (ranges of no chunk when the list is shorter than the workers' shares) the
// pieces are walked worker by worker, skipping the empty ranges.
constexpr int kMergeBatch = 16;

// kSub warps per head: with segments of many pieces (few segments against
// many workers) they take turns over the batches and their states are
// combined in shared memory at the end, in sub-warp order.
template <int kSub>
__global__ void __launch_bounds__(kSub == 1 ? 32 * PKV_MAX_GROUP : 32 * kSub) splitk_merge_kernel(const DecodeArgs a)
{
    __shared__ uint32_t pre_s[kMaxSplitCtas + 1];
    __shared__ __align__(16) float red_a[kSub > 1 ? kSub : 1][32 * 4];   // read and written as float4
    __shared__ float red_ml[kSub > 1 ? kSub : 1][2];
    extern __shared__ float4 merge_stage[];      // [warps][kMergeBatch][32]: the batches' accumulators
    const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // kSub = 1: one CTA per segment, warp g merges query head g; else one CTA
    // per (segment, head g), its kSub warps taking turns over the batches
    const int seg = kSub == 1 ? blockIdx.x : blockIdx.x / a.group;
    const int g = kSub == 1 ? wi : blockIdx.x % a.group, sub = kSub == 1 ? 0 : wi;
    const int b = seg / a.hkv, h = seg % a.hkv;
    const int rank = h * a.batch + b;            // the segment's rank in list order (head-major)

    const float vsc = __ldg(a.v_scale + h);
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the decode grid has finished
    const SegRecord r = a.segs[seg];
    const DecodeHeader hd = *a.header;
    if (r.n <= 0 || r.w0 < 0)
        return;   // empty (the decode kernel wrote its zero rows) or one piece (its worker wrote the output)
    const int64_t total = hd.total, start = r.start;
    const int n_seg = r.n, w0 = r.w0, w1 = r.w1;
    const Split sp = make_split(a, pre_s);

    // every range holds at least one chunk-head when T * wmin >= CT
    const bool dense = total * (a.split ? a.split_wmin : 1) >= sp.ct;
    const bool walk = !dense;
    if (walk && a.split) {                       // the walk reads the split's weight prefix sums
        for (int c = threadIdx.x; c <= a.num_ctas; c += blockDim.x)
            pre_s[c] = g_split_prefix[c];
        __syncthreads();
    }
    const int n_known = w1 - w0 + 1;
    // walk state: worker w, its range [lo_w, hi_w), offset k of the next piece in it
    const int64_t end = start + n_seg;
    int w = w0;
    int64_t lo_w = 0, hi_w = 0, k = 0;
    if (walk) {
        lo_w = range_lo(sp, total, w);
        hi_w = range_lo(sp, total, w + 1);
        k = start - lo_w;
    }

    float M = -INFINITY, L = 0.f;
    float A[4] = {0.f, 0.f, 0.f, 0.f};
    float4 *stage = merge_stage + wi * (kMergeBatch * 32) + lane;   // this lane's [kMergeBatch] entries, 32 apart
    // the walk (empty ranges in the list) is sequential: sub-warp 0 alone
    for (int i0 = sub * kMergeBatch; walk ? sub == 0 : true; i0 += kSub * kMergeBatch) {
        // slot of piece i0 + lane (lanes >= the batch size: -1)
        int my_slot = -1;
        int nb;
        if (!walk) {
            nb = min(kMergeBatch, n_known - i0);
            if (nb <= 0)
                break;
            if (lane < nb)
                my_slot = w0 + i0 + lane;
        } else {
            nb = 0;
            while (nb < kMergeBatch && lo_w + k < end) {
                if (lane == nb)
                    my_slot = w;
                ++nb;
                do {                                                 // next worker with chunks: starts at its range start
                    ++w;
                    lo_w = hi_w;
                    hi_w = range_lo(sp, total, w + 1);
                } while (hi_w <= lo_w && lo_w < end);
                k = 0;
            }
            if (nb == 0)
                break;
        }
        const bool bad = my_slot >= 0 && static_cast<int64_t>(my_slot) + rank >= a.num_slots;
        if (bad)
            my_slot = -1;                                           // skipped, flagged below
        float m = -INFINITY, l = 0.f;
        if (my_slot >= 0) {
            const float *p = a.partials + (static_cast<int64_t>(my_slot + rank) * a.group + g) * kPartialStride;
            m = p[kHeadDim];
            l = p[kHeadDim + 1];
        }
        // This lane's 4 dims of the batch's accumulators, staged in shared
        // memory by asynchronous copies that are all in flight together (one
        // round trip per batch, however the loop is scheduled); pieces past
        // the batch (slot -1) are zero-filled.  Each lane reads back only
        // what it staged.
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
            const int si = __shfl_sync(kFull, my_slot, i);
            const float *src =
                a.partials + (static_cast<int64_t>(si >= 0 ? si + rank : 0) * a.group + g) * kPartialStride + 4 * lane;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(stage + 32 * i)), "l"(src),
                         "r"(si >= 0 ? 16 : 0)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (__any_sync(kFull, bad) && lane == 0 && a.err)
            atomicOr(a.err, PKV_DEVERR_INTERNAL);
        float mb = m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o));
        const float mn = fmaxf(M, mb);
        const float r0 = ex2_approx(M - mn);                     // 0 on the first batch (M = -inf)
        const float sc = my_slot >= 0 ? ex2_approx(m - mn) : 0.f;
        float ls = sc * l;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ls += __shfl_xor_sync(kFull, ls, o);
        L = L * r0 + ls;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            A[c] *= r0;
        asm volatile("cp.async.wait_group 0;" ::: "memory");
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
            const float si = __shfl_sync(kFull, sc, i);
            const float4 v = stage[32 * i];
            A[0] += si * v.x;
            A[1] += si * v.y;
            A[2] += si * v.z;
            A[3] += si * v.w;
        }
        M = mn;
    }
    if constexpr (kSub > 1) {
        *reinterpret_cast<float4 *>(&red_a[wi][4 * lane]) = make_float4(A[0], A[1], A[2], A[3]);
        if (lane == 0) {
            red_ml[wi][0] = M;
            red_ml[wi][1] = L;
        }
        __syncthreads();
        if (sub != 0)
            return;
        float Mt = M;
#pragma unroll
        for (int s2 = 1; s2 < kSub; ++s2)
            Mt = fmaxf(Mt, red_ml[wi + s2][0]);
        const float r0 = ex2_approx(M - Mt);
        L *= r0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            A[c] *= r0;
#pragma unroll
        for (int s2 = 1; s2 < kSub; ++s2) {
            const float ms = red_ml[wi + s2][0];
            const float rs = ms == -INFINITY ? 0.f : ex2_approx(ms - Mt);   // a sub-warp with no pieces adds nothing
            const float4 as = *reinterpret_cast<const float4 *>(&red_a[wi + s2][4 * lane]);
            L += red_ml[wi + s2][1] * rs;
            A[0] += as.x * rs;
            A[1] += as.y * rs;
            A[2] += as.z * rs;
            A[3] += as.w * rs;
        }
    }
    const float f = vsc / L;
    const int64_t row = static_cast<int64_t>(b) * a.hq + static_cast<int64_t>(h) * a.group + g;
    store_pair(a, row, 4 * lane, A[0] * f, A[1] * f);
    store_pair(a, row, 4 * lane + 2, A[2] * f, A[3] * f);
}

}  // namespace

size_t decode_smem_bytes(int /*page_size*/, int batch)
{
    return Smem::bytes(batch);
}

const void *decode_kernel_for(int /*page_size*/)
{
    return reinterpret_cast<const void *>(&paged_gqa_decode_kernel);
}

// Dynamic shared memory of a merge CTA with `warps` warps: the staged batch
// (8 KB a warp).
static size_t merge_stage_bytes(int warps)
{
    return static_cast<size_t>(warps) * kMergeBatch * 32 * sizeof(float4);
}

static std::mutex g_merge_mu;
static bool g_merge_attr[64];   // per device: the merge kernel's shared-memory limit is raised

cudaError_t launch_paged_decode(const DecodeArgs &a, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                int page_size, cudaStream_t stream, const char **site)
{
    const size_t smem = decode_smem_bytes(page_size, a.batch);
    *site = "decode kernel launch";
    paged_gqa_decode_kernel<<<a.num_ctas, kThreads, smem, stream>>>(tm_k, tm_v, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    *site = "split-K merge kernel launch";
    cudaLaunchConfig_t cfg = {};
    // One warp per query head (one CTA per segment) while the segments average
    // fewer than 16 pieces; else one CTA per (segment, query head) whose 2
    // warps (from 16 pieces) or 4 (from 48: few long segments against many
    // workers) take turns over the batches of 16 pieces.
    const int segs = a.batch * a.hkv;
    const long long workers = static_cast<long long>(a.num_ctas) * kWarps;
    const int sub = workers >= 48ll * segs ? 4 : (workers >= 16ll * segs ? 2 : 1);
    const int warps = sub == 1 ? a.group : sub;
    cfg.gridDim = dim3(static_cast<unsigned>(sub == 1 ? segs : segs * a.group), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(32 * warps), 1, 1);
    cfg.dynamicSmemBytes = merge_stage_bytes(warps);
    {
        int dev = -1;
        cudaError_t e2 = cudaGetDevice(&dev);
        if (e2 != cudaSuccess)
            return e2;
        if (dev < 0 || dev >= 64)
            return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lk(g_merge_mu);
        if (!g_merge_attr[dev]) {                // one warp per head of a group of up to 8: up to 64 KB
            *site = "cudaFuncSetAttribute (merge shared memory)";
            e2 = cudaFuncSetAttribute(splitk_merge_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(merge_stage_bytes(PKV_MAX_GROUP)));
            if (e2 != cudaSuccess)
                return e2;
            g_merge_attr[dev] = true;
            *site = "split-K merge kernel launch";
        }
    }
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (sub == 4)
        return cudaLaunchKernelEx(&cfg, splitk_merge_kernel<4>, a);
    return sub == 2 ? cudaLaunchKernelEx(&cfg, splitk_merge_kernel<2>, a) : cudaLaunchKernelEx(&cfg, splitk_merge_kernel<1>, a);
}

cudaError_t upload_split_prefix(const uint32_t *prefix, int n)
{
    if (n < 1 || n > kMaxSplitCtas)
        return cudaErrorInvalidValue;
    return cudaMemcpyToSymbol(g_split_prefix, prefix, (static_cast<size_t>(n) + 1) * sizeof(uint32_t));
}

cudaError_t clear_split_probe(int n, cudaStream_t stream)
{
    if (n < 1 || n > kMaxSplitCtas)
        return cudaErrorInvalidValue;
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_split_probe);
    if (e != cudaSuccess)
        return e;
    return cudaMemsetAsync(p, 0, static_cast<size_t>(n) * 2 * sizeof(unsigned long long), stream);
}

cudaError_t read_split_probe(unsigned long long *times, int n)
{
    if (n < 1 || n > kMaxSplitCtas)
        return cudaErrorInvalidValue;
    return cudaMemcpyFromSymbol(times, g_split_probe, static_cast<size_t>(n) * 2 * sizeof(unsigned long long));
}

}  // namespace pkv
