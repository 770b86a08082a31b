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
// list of "page-heads" (one page of one kv head, 2 x P x 128 bytes).  Each of
// C persistent CTAs takes an equal contiguous range of that list, whatever
// the sequence lengths (flash-decoding split-K with perfect balance).  A CTA
// range cuts segments into pieces; a piece that covers a whole segment writes
// the final output, the others write a partial softmax state (running max m,
// sum l, unnormalised accumulator) into workspace slot (cta + segment), and
// a second small kernel merges the pieces of each segment in CTA order.
//
// Inside a CTA: one producer warp walks the CTA's pages, fetches block-table
// entries 32 at a time one batch ahead, and issues two TMA tensor loads per
// page (K tile, V tile; 128-byte swizzled, evict-first in L2) into an
// 8-stage shared-memory ring guarded by full/empty mbarriers.  Four consumer
// warps take the pages round-robin.  Each warp reads a 16-token tile with
// ldmatrix (conflict-free thanks to the swizzle), widens E4M3 to f16 exactly
// in registers, and runs both products on the tensor cores with mma.sync
// m16n8k16 (f16 in, f32 accumulate):
//   S[g][t]   = Q[g][:] . K[t][:]    (A = Q, the group's <= 8 heads; B = K)
//   O^T[d][g] += V^T[d][t] P^T[t][g]  (A = V via ldmatrix.trans; B = P)
// The QK^T output fragment is already laid out as the PV B fragment, so the
// probabilities never leave registers.  P is split into f16 hi + lo parts
// (two PV products) so the probabilities keep ~22 significant bits.  The
// online softmax runs in the exp2 domain with a lazy rescale (only when a
// running max grows by more than 2^8).  At the end of a piece the four warps
// merge their states through shared memory.
//
// Every wait on an mbarrier is bounded (2 s on the global timer): on expiry
// the kernel raises PKV_DEVERR_TIMEOUT, stops issuing copies, drains the ones
// in flight and returns.
#include <math.h>

#include "internal.h"

namespace pkv {

namespace {

constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr unsigned kFull = 0xffffffffu;
constexpr int kCombineThreads = 128;

struct Loc {
    int b, h, pg;   // sequence, kv head, page index within the sequence
};

__device__ __forceinline__ int clamp_len(int L, int cap)
{
    return L < 0 ? 0 : (L > cap ? cap : L);
}

__device__ __forceinline__ int pages_of(const int *ps, int b)
{
    return ps[b + 1] - ps[b];
}

// Segment (b, h) covers list positions [ps[b]*hkv + h*np_b, ... + np_b).
__device__ Loc locate(const int *ps, int batch, int hkv, int64_t x)
{
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(ps[mid]) * hkv <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int64_t rem = x - static_cast<int64_t>(ps[lo]) * hkv;
    const int np = pages_of(ps, lo);
    Loc l;
    l.b = lo;
    l.h = static_cast<int>(rem / np);
    l.pg = static_cast<int>(rem % np);
    return l;
}

__device__ Loc advance(const int *ps, int batch, int hkv, Loc l, int64_t n)
{
    int64_t pg = l.pg + n;
    while (l.b < batch) {
        const int np = pages_of(ps, l.b);
        if (pg < np)
            break;
        pg -= np;
        if (++l.h == hkv) {
            l.h = 0;
            ++l.b;
        }
    }
    l.pg = static_cast<int>(pg);
    return l;
}

// CTA whose range holds list position x (ranges are [c*T/C, (c+1)*T/C)).
__device__ __forceinline__ int cta_of(int64_t x, int64_t total, int ctas)
{
    return static_cast<int>(((x + 1) * ctas - 1) / total);
}

template <int P>
struct Smem {
    static constexpr int kTile = P * kHeadDim;              // bytes of one K (or V) tile
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kBar = kStages * kStageBytes;      // full[kStages], empty[kStages]
    static constexpr int kFlag = kBar + 2 * kStages * 8;    // abort flag
    static constexpr int kWarpSum = kFlag + 16;             // scan scratch (5 ints)
    static constexpr int kCm = kWarpSum + 32;               // [warps][8] running max
    static constexpr int kCl = kCm + kConsumerWarps * 8 * 4;        // [warps][8] sums
    static constexpr int kCa = kCl + kConsumerWarps * 8 * 4;        // [warps][8][128] accumulators
    static constexpr int kPstart = kCa + kConsumerWarps * 8 * kHeadDim * 4;
    static_assert(kCa % 16 == 0, "accumulator scratch must be 16-byte aligned");
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

// One 16-token tile: scores, online softmax update, P.V accumulation.
// kt / vt: shared addresses of the tile's K and V rows (128 B each, 128-byte
// swizzle, tile base 1024-byte aligned).  nv: valid tokens in the tile (1..16).
__device__ __forceinline__ void process_tile(uint32_t kt, uint32_t vt, int nv, const uint32_t (&qa)[8][2],
                                             float scale2, float &m_ref, float &lsum, float (&acc)[8][4],
                                             int lane)
{
    const int t4 = lane & 3;
    const int r = lane & 7;
    const int mi = lane >> 3;

    // K fragments: matrix (j, sg) = tokens 8j..8j+7, dims 16sg..16sg+15.
    uint32_t kf[2][8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int j = mi & 1, sg = 2 * q + (mi >> 1), tok = 8 * j + r;
        ldsm_x4(kt + tok * kHeadDim + ((sg ^ r) << 4), kf[0][2 * q], kf[1][2 * q], kf[0][2 * q + 1],
                kf[1][2 * q + 1]);
    }
    // V fragments (transposed): matrix (hh, sg) = tokens 8hh..8hh+7, dims 16sg..16sg+15.
    uint32_t vf[2][8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int hh = mi & 1, sg = 2 * q + (mi >> 1), tok = 8 * hh + r;
        ldsm_x4_trans(vt + tok * kHeadDim + ((sg ^ r) << 4), vf[0][2 * q], vf[1][2 * q],
                      vf[0][2 * q + 1], vf[1][2 * q + 1]);
    }

    // S = Q K^T.  Thread (gid, t4) gets S[head gid][tokens 8j + 2t4, 8j + 2t4 + 1].
    float sc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            sc[j][c] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int j = 0; j < 2; ++j)
            mma_16816(sc[j], qa[kk][0], 0u, qa[kk][1], 0u, e4m3x2_to_f16x2(kf[j][kk]),
                      e4m3x2_to_f16x2(kf[j][kk] >> 16));

    float y[4];
    y[0] = (2 * t4 < nv) ? sc[0][0] * scale2 : -INFINITY;
    y[1] = (2 * t4 + 1 < nv) ? sc[0][1] * scale2 : -INFINITY;
    y[2] = (8 + 2 * t4 < nv) ? sc[1][0] * scale2 : -INFINITY;
    y[3] = (9 + 2 * t4 < nv) ? sc[1][1] * scale2 : -INFINITY;
    float tmax = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
    tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 2));
    if (__any_sync(kFull, tmax > m_ref + kRescaleThreshold)) {
        const float m_new = fmaxf(m_ref, tmax);
        const float alpha = exp2f(m_ref - m_new);
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
    const float p0 = exp2f(y[0] - m_ref), p1 = exp2f(y[1] - m_ref);
    const float p2 = exp2f(y[2] - m_ref), p3 = exp2f(y[3] - m_ref);
    lsum += (p0 + p1) + (p2 + p3);
    const uint32_t h01 = f32x2_to_f16x2(p0, p1), h23 = f32x2_to_f16x2(p2, p3);
    const float2 b01 = f16x2_to_f32x2(h01), b23 = f16x2_to_f32x2(h23);
    const uint32_t l01 = f32x2_to_f16x2(p0 - b01.x, p1 - b01.y);
    const uint32_t l23 = f32x2_to_f16x2(p2 - b23.x, p3 - b23.y);

    if (nv < 16) {   // rows past the sequence end may hold anything (even NaN codes)
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
    for (int sg = 0; sg < 8; ++sg) {
        const uint32_t x0 = __byte_perm(vf[0][sg], 0, 0x3120);
        const uint32_t x1 = __byte_perm(vf[1][sg], 0, 0x3120);
        const uint32_t a0 = e4m3x2_to_f16x2(x0), a1 = e4m3x2_to_f16x2(x0 >> 16);
        const uint32_t a2 = e4m3x2_to_f16x2(x1), a3 = e4m3x2_to_f16x2(x1 >> 16);
        mma_16816(acc[sg], a0, a1, a2, a3, h01, h23);
        mma_16816(acc[sg], a0, a1, a2, a3, l01, l23);
    }
}

template <int P>
__global__ void __launch_bounds__(kThreads, 3)
    paged_gqa_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const DecodeArgs a)
{
    using S = Smem<P>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int *pstart = reinterpret_cast<int *>(smem + S::kPstart);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S::kFlag);
    int *warp_sum = reinterpret_cast<int *>(smem + S::kWarpSum);
    const uint32_t ring = smem_addr(smem);
    const uint32_t bar_full = smem_addr(smem + S::kBar);
    const uint32_t bar_empty = bar_full + 8 * kStages;
    const int cap = a.max_pages * P;

    // ---- per-sequence page offsets (every CTA computes them; B ints from L2)
    {
        const int chunk = (a.batch + kThreads - 1) / kThreads;
        const int b0 = min(a.batch, tid * chunk), b1 = min(a.batch, b0 + chunk);
        int local = 0;
        for (int b = b0; b < b1; ++b)
            local += (clamp_len(__ldg(a.seq_lens + b), cap) + P - 1) / P;
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
            *abort_flag = 0;
            for (int s = 0; s < kStages; ++s) {
                mbar_init(bar_full + 8 * s, 1);
                mbar_init(bar_empty + 8 * s, 1);
            }
            fence_barrier_init();
        }
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w)
            base += warp_sum[w];
        int run = base + incl - local;
        for (int b = b0; b < b1; ++b) {
            const int L = __ldg(a.seq_lens + b);
            pstart[b] = run;
            run += (clamp_len(L, cap) + P - 1) / P;
            if (blockIdx.x == 0 && a.err && (L < 0 || L > cap))
                atomicOr(a.err, PKV_DEVERR_SEQLEN);
        }
        if (tid == kThreads - 1)
            pstart[a.batch] = base + incl;
        __syncthreads();
    }

    const int64_t total = static_cast<int64_t>(pstart[a.batch]) * a.hkv;
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * total / a.num_ctas;
    const int64_t hi = static_cast<int64_t>(blockIdx.x + 1) * total / a.num_ctas;
    if (lo >= hi)
        return;

    if (warp == kConsumerWarps) {
        // ================= producer warp =================
        const uint64_t policy = l2_policy_evict_first();
        const int64_t n_total = hi - lo;
        const int zoob = static_cast<int>(a.num_pages * a.hkv);   // first out-of-pool tile: reads zeros
        auto tile_z = [&](Loc l) -> int {
            const int phys = __ldg(a.block_table + static_cast<int64_t>(l.b) * a.max_pages + l.pg);
            if (phys < 0 || phys >= a.num_pages) {
                if (a.err)
                    atomicOr(a.err, PKV_DEVERR_PAGE);
                return zoob;
            }
            return phys * a.hkv + l.h;
        };
        Loc base = locate(pstart, a.batch, a.hkv, lo);
        int my_z = 0;
        if (lane < n_total)
            my_z = tile_z(advance(pstart, a.batch, a.hkv, base, lane));
        int64_t issued = 0;
        for (int64_t i0 = 0; i0 < n_total; i0 += 32) {
            const int n = static_cast<int>(min(static_cast<int64_t>(32), n_total - i0));
            const Loc next = advance(pstart, a.batch, a.hkv, base, 32);
            int next_z = 0;
            if (i0 + 32 + lane < n_total)
                next_z = tile_z(advance(pstart, a.batch, a.hkv, next, lane));
            for (int j = 0; j < n; ++j) {
                const int z = __shfl_sync(kFull, my_z, j);
                if (lane == 0 && !*abort_flag) {
                    const int64_t i = i0 + j;
                    const int s = static_cast<int>(i % kStages);
                    const uint32_t u = static_cast<uint32_t>(i / kStages);
                    bool ok = true;
                    if (u > 0)
                        ok = wait_thread(bar_empty + 8 * s, (u - 1) & 1u, abort_flag, a.err, true);
                    if (ok) {
                        const uint32_t dst = ring + s * S::kStageBytes;
                        mbar_arrive_expect_tx(bar_full + 8 * s, 2 * S::kTile);
                        tma_load_3d(dst, &tm_k, 0, 0, z, bar_full + 8 * s, policy);
                        tma_load_3d(dst + S::kTile, &tm_v, 0, 0, z, bar_full + 8 * s, policy);
                        issued = i + 1;
                    }
                }
            }
            my_z = next_z;
            base = next;
        }
        // Drain: never leave the CTA with a copy still writing shared memory.
        if (lane == 0) {
            for (int s = 0; s < kStages && s < issued; ++s) {
                const uint32_t u = static_cast<uint32_t>((issued - 1 - s) / kStages);
                wait_thread(bar_full + 8 * s, u & 1u, abort_flag, a.err, false);
            }
        }
        return;
    }

    // ================= consumer warps =================
    const int gid = lane >> 2, t4 = lane & 3;
    float *cm = reinterpret_cast<float *>(smem + S::kCm);
    float *cl = reinterpret_cast<float *>(smem + S::kCl);
    float *ca = reinterpret_cast<float *>(smem + S::kCa);
    Loc loc = locate(pstart, a.batch, a.hkv, lo);
    int64_t cur = lo, ibase = 0;
    while (cur < hi) {
        const int np = pages_of(pstart, loc.b);
        const int n_piece = static_cast<int>(min(static_cast<int64_t>(np - loc.pg), hi - cur));
        const int L = clamp_len(__ldg(a.seq_lens + loc.b), cap);
        const bool whole = (loc.pg == 0) && (n_piece == np);
        const int seg = loc.b * a.hkv + loc.h;
        const float scale2 = __ldg(a.k_scale + loc.h) * a.sm_scale_log2;

        // Q fragment for k-step kk: head gid, dims 16kk + 4t4 + {0,1} and {2,3}.
        uint32_t qa[8][2];
        {
            const bool valid = gid < a.group;
            const __nv_bfloat16 *qrow =
                a.q + (static_cast<int64_t>(loc.b) * a.hq + loc.h * a.group + (valid ? gid : 0)) * kHeadDim;
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
#pragma unroll
        for (int sg = 0; sg < 8; ++sg)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                acc[sg][c] = 0.f;

        const int64_t iend = ibase + n_piece;
        for (int64_t i = ibase + (warp - ibase % kConsumerWarps + kConsumerWarps) % kConsumerWarps; i < iend;
             i += kConsumerWarps) {
            const int page = loc.pg + static_cast<int>(i - ibase);
            const int nv = min(P, L - page * P);
            const int s = static_cast<int>(i % kStages);
            const uint32_t par = static_cast<uint32_t>(i / kStages) & 1u;
            if (!wait_warp(bar_full + 8 * s, par, abort_flag, a.err, lane))
                continue;
            const uint32_t kt = ring + s * S::kStageBytes;
#pragma unroll
            for (int sub = 0; sub < P / 16; ++sub)
                if (sub * 16 < nv)
                    process_tile(kt + sub * 16 * kHeadDim, kt + S::kTile + sub * 16 * kHeadDim, nv - sub * 16,
                                 qa, scale2, m_ref, lsum, acc, lane);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_empty + 8 * s);
        }

        // ---- merge the four warps' states of this piece
        lsum += __shfl_xor_sync(kFull, lsum, 1);
        lsum += __shfl_xor_sync(kFull, lsum, 2);
        if (t4 == 0) {
            cm[warp * 8 + gid] = m_ref;
            cl[warp * 8 + gid] = lsum;
        }
#pragma unroll
        for (int sg = 0; sg < 8; ++sg) {
            const int d = 16 * sg + 2 * gid;
            *reinterpret_cast<float2 *>(ca + (warp * 8 + 2 * t4) * kHeadDim + d) = make_float2(acc[sg][0], acc[sg][2]);
            *reinterpret_cast<float2 *>(ca + (warp * 8 + 2 * t4 + 1) * kHeadDim + d) =
                make_float2(acc[sg][1], acc[sg][3]);
        }
        named_barrier(1, kConsumerWarps * 32);
        const float vsc = __ldg(a.v_scale + loc.h);
        const int64_t row0 = static_cast<int64_t>(loc.b) * a.hq + loc.h * a.group;
        for (int e = tid; e < a.group * kHeadDim; e += kConsumerWarps * 32) {
            const int g = e >> 7, d = e & (kHeadDim - 1);
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w)
                M = fmaxf(M, cm[w * 8 + g]);
            float Ls = 0.f, A = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = exp2f(cm[w * 8 + g] - M);
                Ls += cl[w * 8 + g] * f;
                A += ca[(w * 8 + g) * kHeadDim + d] * f;
            }
            if (whole) {
                store_out(a, row0 + g, d, A / Ls * vsc);
            } else {
                float *slot = a.partials +
                              (static_cast<int64_t>(blockIdx.x + seg) * a.group + g) * kPartialStride;
                slot[d] = A;
                if (d == 0) {
                    slot[kHeadDim] = M;
                    slot[kHeadDim + 1] = Ls;
                }
            }
        }
        named_barrier(1, kConsumerWarps * 32);

        cur += n_piece;
        ibase += n_piece;
        loc = advance(pstart, a.batch, a.hkv, loc, n_piece);
    }
}

// Merges the pieces of every segment that more than one CTA touched, writes
// zeros for empty sequences, and leaves single-piece segments alone.
__global__ void __launch_bounds__(kCombineThreads) splitk_combine_kernel(const DecodeArgs a, int P)
{
    __shared__ int red[2][kCombineThreads / 32];
    const int seg = blockIdx.x;
    const int b = seg / a.hkv, h = seg % a.hkv;
    const int cap = a.max_pages * P;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int before = 0, all = 0;
    for (int bb = threadIdx.x; bb < a.batch; bb += kCombineThreads) {
        const int np = (clamp_len(__ldg(a.seq_lens + bb), cap) + P - 1) / P;
        all += np;
        if (bb < b)
            before += np;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(kFull, before, o);
        all += __shfl_xor_sync(kFull, all, o);
    }
    if (lane == 0) {
        red[0][warp] = before;
        red[1][warp] = all;
    }
    __syncthreads();
    before = 0;
    all = 0;
#pragma unroll
    for (int w = 0; w < kCombineThreads / 32; ++w) {
        before += red[0][w];
        all += red[1][w];
    }
    const int np = (clamp_len(__ldg(a.seq_lens + b), cap) + P - 1) / P;
    const int64_t row0 = static_cast<int64_t>(b) * a.hq + static_cast<int64_t>(h) * a.group;
    if (np == 0) {
        for (int e = threadIdx.x; e < a.group * kHeadDim; e += kCombineThreads)
            store_out(a, row0 + (e >> 7), e & (kHeadDim - 1), 0.f);
        return;
    }
    const int64_t total = static_cast<int64_t>(all) * a.hkv;
    const int64_t start = static_cast<int64_t>(before) * a.hkv + static_cast<int64_t>(h) * np;
    const int c0 = cta_of(start, total, a.num_ctas);
    const int c1 = cta_of(start + np - 1, total, a.num_ctas);
    if (c0 == c1)
        return;
    const float vsc = __ldg(a.v_scale + h);
    // CTAs between c0 and c1 whose range is empty (more CTAs than page-heads)
    // wrote nothing: skip their slots.
    auto has_piece = [&](int c) {
        return static_cast<int64_t>(c) * total / a.num_ctas != static_cast<int64_t>(c + 1) * total / a.num_ctas;
    };
    for (int e = threadIdx.x; e < a.group * kHeadDim; e += kCombineThreads) {
        const int g = e >> 7, d = e & (kHeadDim - 1);
        float M = -INFINITY;
        for (int c = c0; c <= c1; ++c)
            if (has_piece(c))
                M = fmaxf(M, a.partials[(static_cast<int64_t>(c + seg) * a.group + g) * kPartialStride + kHeadDim]);
        float Ls = 0.f, A = 0.f;
        for (int c = c0; c <= c1; ++c) {
            if (!has_piece(c))
                continue;
            const float *slot = a.partials + (static_cast<int64_t>(c + seg) * a.group + g) * kPartialStride;
            const float f = exp2f(slot[kHeadDim] - M);
            Ls += slot[kHeadDim + 1] * f;
            A += slot[d] * f;
        }
        store_out(a, row0 + g, d, A / Ls * vsc);
    }
}

template <int P>
const void *decode_kernel_ptr()
{
    return reinterpret_cast<const void *>(&paged_gqa_decode_kernel<P>);
}

}  // namespace

size_t decode_smem_bytes(int page_size, int batch)
{
    return page_size == 32 ? Smem<32>::bytes(batch) : Smem<16>::bytes(batch);
}

const void *decode_kernel_for(int page_size)
{
    return page_size == 32 ? decode_kernel_ptr<32>() : decode_kernel_ptr<16>();
}

cudaError_t launch_paged_decode(const DecodeArgs &a, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                int page_size, cudaStream_t stream)
{
    const size_t smem = decode_smem_bytes(page_size, a.batch);
    if (a.num_ctas > 0) {
        if (page_size == 32)
            paged_gqa_decode_kernel<32><<<a.num_ctas, kThreads, smem, stream>>>(tm_k, tm_v, a);
        else
            paged_gqa_decode_kernel<16><<<a.num_ctas, kThreads, smem, stream>>>(tm_k, tm_v, a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    splitk_combine_kernel<<<a.batch * a.hkv, kCombineThreads, 0, stream>>>(a, page_size);
    return cudaGetLastError();
}

}  // namespace pkv
