// MLA paged decode attention kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// Absorbed MLA decode is MQA with one KV head: key [ckv | kpe] (576), value
// ckv (512) ("Benchmarking MLA", FlashInfer issue #700).  Each CTA owns HG query
// heads of every (request, token range) segment in its slot of the plan and
// walks the segment in 128-token tiles.  Both contractions are computed
// transposed, so that the 128-row UMMA M dimension is filled by tokens (or
// latent dims) even when only 16 heads exist:
//
//   S^T[t, h]  = sum_k K[t, k] * Q[h, k]        (M = 128 tokens, N = HG, K = 576)
//   O^T[d, h] += sum_t V[t, d] * P[h, t]        (M = 128 dims x 4, N = HG, K = 128 tokens)
//
// Accumulators live in TMEM (lane = token for S^T, lane = latent dim for O^T):
// two S^T buffers of HG columns and O^T in 4*HG columns.
//
// A tcgen05.mma costs at least ~64 SM cycles whatever its size, so with N = 16
// the token rate is set by the instruction count: 36 score + 32 PV MMAs per
// 128 tokens, which needs 128-token tiles.  A tile of ckv+kpe is 144 KB, too
// large to double-buffer in shared memory, so it is held in small slots that
// are released piece by piece: a 16 KB kpe slot (freed once the score MMA has
// read it) and four 32 KB ckv "pair" slots (two 64-dim chunks = one 128-dim M
// block of O^T), each read by the score MMA and freed when the PV MMA of its
// block completes.  With one pair slot more than a tile needs, the score MMA
// of tile j+1 starts while the softmax of tile j runs, and every PV block of
// tile j frees the slot that tile j+1's next block loads into.  Each KV byte
// enters the SM once.  The ring is too shallow to cover DRAM latency under
// full load (about 3 us, ~130 KB per SM in flight), so the producer also
// prefetches the pages of the tile two ahead into L2 with
// cp.async.bulk.prefetch, which needs no shared memory; the ring then only
// covers L2 latency.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q^T once per segment, L2 prefetch two tiles
//               ahead, then per tile the kpe rows and the 4 ckv pairs of every
//               page (128-byte swizzle).  For a request's last, partial tile it
//               zeroes the rows past the last token (stale or NaN bytes) in the
//               pair slots before publishing them.
//   warp 1      TMEM allocation; one thread issues every tcgen05.mma, picking
//               whichever is ready of the next score block (tile j+1) and the
//               next PV block (tile j).
//   warps 2..5  softmax + epilogue: thread i owns TMEM lane i (token i of the
//               tile for S^T, latent dims i + 128c for O^T).
//
// Online softmax (log2 domain) with a lazily updated running max: a head's
// max is only moved (and O^T and the partial row sums rescaled) when the tile
// max exceeds it by more than 8 (a factor 256); the final normalisation uses
// the same max for O and l, so the result is exact up to rounding.  P is
// rounded to bf16 for the PV MMA.
//
// Split-KV merge (FlashMLA PR #233, "deterministic combine"): a piece of a
// split request writes its normalised partial (o, lse); the CTA whose arrival
// on the request's counter is the last one merges all pieces in slot order
//   M = max_i lse_i, w_i = exp(lse_i - M), out = sum_i w_i o_i / sum_i w_i,
//   lse = M + ln sum_i w_i,
// and resets the counter for the next run.  The arithmetic does not depend on
// which CTA merges, so results are bit-identical from run to run.
//
// Every mbarrier wait is bounded; on expiry the kernel records a status code,
// drains its in-flight copies and MMAs, frees TMEM and returns.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "plan.h"
#include "ptx.cuh"

namespace mla {

constexpr uint32_t kStatusTimeout = 0x100u;       // OR-ed with the wait site id
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s without progress before giving up

struct AttnParams {
    const int32_t* unit_ptr;      // [num_units + 1]
    const Segment* segments;      // [num_segments]
    const int32_t* kv_indices;
    const int32_t* kv_indptr;
    const uint8_t* ckv;           // cache base addresses (L2 prefetch of whole pages)
    const uint8_t* kpe;
    float* out;                   // [B, h_q, 512]
    float* lse;                   // [B, h_q]
    float* part_o;                // [num_partials, h_q, 512]
    float* part_lse;              // [num_partials, h_q]
    const float* ckv_scale;       // e4m3 cache: fp32 scale per token [num_pages * page_size], else null
    int32_t* counters;            // arrivals per (split request, 16- or 32-head block)
    uint32_t* status;
    uint64_t* trace;              // per-tile event timestamps when built with MLA_TRACE, else unused
    float scale_log2;             // sm_scale * log2(e)
    int h_q;
    int page_size;
    int head_groups;
};

template <int HG>
struct AttnCfg {
    static_assert(HG == 16 || HG == 32, "heads per CTA");
    static constexpr int kThreads = 192;
    static constexpr int kSoftmaxThreads = 128;
    static constexpr int kQBufs = (HG == 16) ? 2 : 1;
    static constexpr int kPBufs = (HG == 16) ? 2 : 1;
    static constexpr int kPairSlots = 5;
    static constexpr int kKpeSlots = 1;
    static constexpr int kPrefetchTiles = 2;   // pages of tile j + 2 are prefetched into L2 while tile j loads
    static constexpr int kChunkBytes = kTileTokens * 128;      // 64 dims x 128 tokens bf16 = 16 KB
    static constexpr int kPairBytes = 2 * kChunkBytes;         // 32 KB
    static constexpr int kQChunkBytes = HG * 128;              // 64 dims x HG heads
    static constexpr int kQBytes = 9 * kQChunkBytes;
    static constexpr int kQStride = ((kQBytes + 1023) / 1024) * 1024;
    static constexpr int kPChunkBytes = HG * 128;              // 64 tokens x HG heads
    static constexpr int kPStride = ((2 * kPChunkBytes + 1023) / 1024) * 1024;

    static constexpr int kOffPair = 0;
    static constexpr int kOffKpe = kOffPair + kPairSlots * kPairBytes;
    static constexpr int kOffQ = kOffKpe + kKpeSlots * kChunkBytes;
    static constexpr int kOffP = kOffQ + kQBufs * kQStride;
    static constexpr int kOffMisc = kOffP + kPBufs * kPStride;
    static constexpr int kMiscBytes = 3072;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");

    // TMEM columns: S^T buffer b at b*HG, O^T block c at 64 + c*HG
    static constexpr uint32_t kTmemO = 64;
    static constexpr uint32_t kTmemCols = (kTmemO + 4 * HG <= 128) ? 128 : 256;

    static constexpr uint32_t kIdescS = idesc_bf16(128, HG, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16(128, HG, true, false);
};

struct AttnMisc {
    uint64_t q_full[2], q_empty[2], s_full[2], p_full[2], pv_done, o_full, drain;
    uint64_t kfull[1], kempty[1];
    uint64_t pfull[5], pempty[5], pload[5];
    uint32_t tmem_base;
    int abort_flag;
    int merge_flag;
    float red_max[2][4][32];
    float red_sum[4][32];
    float mrg_max[32];
    float mrg_inv[32];
    float mrg_w[8 * 32];
};

static_assert(sizeof(AttnMisc) <= 3072, "misc region");

// Bounded wait on an mbarrier phase.  Returns false if the kernel is aborting
// (abort_flag set by another warp) or after kWaitLimitNs without completion, in which
// case it sets abort_flag and records `site` in the status word.
__device__ __forceinline__ bool wait_phase_flag(uint64_t* bar, uint32_t parity, int* abort_flag, uint32_t* status,
                                                uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *reinterpret_cast<volatile int*>(abort_flag) = 1;
            atomicCAS(status, 0u, kStatusTimeout | site);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, AttnMisc* misc, uint32_t* status,
                                           uint32_t site) {
    return wait_phase_flag(bar, parity, &misc->abort_flag, status, site);
}

// Optional pipeline timeline (compiled in with -DMLA_TRACE): CTAs 0..3 record the
// global timer at event `ev` of their tile `idx` into prm.trace[cta][ev][idx].
#ifdef MLA_TRACE
#define MLA_TRACE_EVENT(ev, idx)                                                              \
    do {                                                                                      \
        if (prm.trace && blockIdx.x < 2 && (idx) < 256)                                       \
            prm.trace[(blockIdx.x * 8 + (ev)) * 256 + (idx)] = global_timer_ns();            \
    } while (0)
// CTA 0 only: a timestamp per unit of work (a ring slot fill, ...) in the area of CTAs 2 and 3,
// lane `ln` (0..3) of 1024 entries each.
#define MLA_TRACE_UNIT(ln, idx)                                                               \
    do {                                                                                      \
        if (prm.trace && blockIdx.x == 0 && (idx) < 1024)                                     \
            prm.trace[2 * 8 * 256 + (ln) * 1024 + (idx)] = global_timer_ns();                 \
    } while (0)
// Every CTA also records 8 milestones (entry, producer done, ...) after the per-tile area.
#define MLA_TRACE_CTA(k)                                                                      \
    do {                                                                                      \
        if (prm.trace) prm.trace[4 * 8 * 256 + blockIdx.x * 8 + (k)] = global_timer_ns();     \
    } while (0)
#else
#define MLA_TRACE_EVENT(ev, idx) \
    do {                         \
    } while (0)
#define MLA_TRACE_CTA(k) \
    do {                 \
    } while (0)
#define MLA_TRACE_UNIT(ln, idx) \
    do {                        \
    } while (0)
#endif

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Merge of the split pieces of one request for heads [head0, head0 + NH), run by the CTA
// whose piece arrived last (FlashMLA PR #233, "deterministic combine"): with lse_i the
// natural-log partial lse of piece i and o_i its normalised partial output,
//     M = max_i lse_i,  w_i = exp(lse_i - M) / sum_j exp(lse_j - M),
//     out = sum_i w_i o_i,  lse = M + ln sum_j exp(lse_j - M).
// Every sum runs in a fixed order (pieces in slot order, fixed shuffle trees), so reruns
// give identical bits.  The loads are issued in batches (all heads of a piece at once) so
// the merge costs a few memory round trips rather than one per (piece, head).
// NTHR threads (tid 0..NTHR-1) call it together and synchronise on named barrier `bar`.
// Scratch in shared memory: s_max[NH], s_inv[NH], s_w[NTHR] (NTHR >= 8 * 16).
template <int NH, int NTHR>
__device__ __forceinline__ void merge_split_pieces(const AttnParams& prm, int b, int slot_begin, int n_slots,
                                                   int head0, int tid, uint32_t bar, float* s_max, float* s_inv,
                                                   float* s_w) {
    static_assert(NTHR == 128 && NH % 16 == 0 && NTHR % NH == 0, "merge layout");
    constexpr int kTph = NTHR / NH;    // threads per head in the lse pass
    constexpr int kChunk = NTHR / 16;  // pieces whose weights are staged at a time (8)
    const size_t hq = static_cast<size_t>(prm.h_q);
    {
        // ---- lse pass: thread (h, sub) scans pieces sub, sub + kTph, ... with a running (max, sum)
        const int h = tid / kTph, sub = tid % kTph;
        float m = -INFINITY, s = 0.f;
        for (int i = sub; i < n_slots; i += kTph) {
            const float x = __ldcg(prm.part_lse + (slot_begin + i) * hq + head0 + h);
            if (x > m) {
                s = (m == -INFINITY ? 0.f : s * expf(m - x)) + 1.f;
                m = x;
            } else {
                s += expf(x - m);
            }
        }
#pragma unroll
        for (int o = kTph / 2; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            const float mm = fmaxf(m, m2);
            const float a = (m == -INFINITY) ? 0.f : s * expf(m - mm);
            const float c = (m2 == -INFINITY) ? 0.f : s2 * expf(m2 - mm);
            s = a + c;   // both lanes of the pair add the same two values (addition commutes exactly)
            m = mm;
        }
        if (sub == 0) {
            s_max[h] = m;
            s_inv[h] = 1.f / s;
            prm.lse[static_cast<size_t>(b) * hq + head0 + h] = m + logf(s);
        }
    }
    named_barrier_sync(bar, NTHR);
    // ---- outputs: thread tid owns dims [4 tid, 4 tid + 4) of every head
    float4* out4 = reinterpret_cast<float4*>(prm.out + (static_cast<size_t>(b) * hq + head0) * kDimCkv) + tid;
#pragma unroll 1
    for (int hb = 0; hb < NH; hb += 16) {
        float4 acc[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int c0 = 0; c0 < n_slots; c0 += kChunk) {
            {
                const int i = tid / 16, h = tid % 16;   // weight of piece c0 + i for head hb + h
                float w = 0.f;
                if (c0 + i < n_slots)
                    w = expf(__ldcg(prm.part_lse + (slot_begin + c0 + i) * hq + head0 + hb + h) - s_max[hb + h]) *
                        s_inv[hb + h];
                s_w[tid] = w;
            }
            named_barrier_sync(bar, NTHR);
            const int n = min(kChunk, n_slots - c0);
#pragma unroll 1
            for (int i = 0; i < n; ++i) {
                const float4* src =
                    reinterpret_cast<const float4*>(prm.part_o + ((slot_begin + c0 + i) * hq + head0 + hb) * kDimCkv) + tid;
                float4 v[16];
#pragma unroll
                for (int h = 0; h < 16; ++h) v[h] = __ldcg(src + h * (kDimCkv / 4));
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    const float w = s_w[i * 16 + h];
                    acc[h].x = fmaf(w, v[h].x, acc[h].x);
                    acc[h].y = fmaf(w, v[h].y, acc[h].y);
                    acc[h].z = fmaf(w, v[h].z, acc[h].z);
                    acc[h].w = fmaf(w, v[h].w, acc[h].w);
                }
            }
            named_barrier_sync(bar, NTHR);   // s_w is rewritten next
        }
#pragma unroll
        for (int h = 0; h < 16; ++h) out4[(hb + h) * (kDimCkv / 4)] = acc[h];
    }
}

// Walks the non-empty segments of one CTA slot tile by tile.
template <int TILE>
struct TileCursorT {
    const Segment* segs;
    int si, end;
    Segment sg;
    int t0;
    __device__ __forceinline__ bool next_segment() {
        for (++si; si < end; ++si) {
            sg = segs[si];
            if (sg.t_end > sg.t_begin) {
                t0 = sg.t_begin;
                return true;
            }
        }
        return false;
    }
    __device__ __forceinline__ bool init(const Segment* s, int begin, int e) {
        segs = s;
        si = begin - 1;
        end = e;
        return next_segment();
    }
    // advance by one tile; returns false at the end of the slot, sets new_seg on a segment change
    __device__ __forceinline__ bool advance(bool& new_seg) {
        t0 += TILE;
        new_seg = false;
        if (t0 < sg.t_end) return true;
        new_seg = true;
        return next_segment();
    }
    __device__ __forceinline__ bool first() const { return t0 == sg.t_begin; }
    __device__ __forceinline__ bool last() const { return t0 + TILE >= sg.t_end; }
    __device__ __forceinline__ int ntok() const { return min(TILE, sg.t_end - t0); }
};
using TileCursor = TileCursorT<kTileTokens>;

template <int HG>
__global__ void __launch_bounds__(AttnCfg<HG>::kThreads, 1)
    mla_decode_attn_kernel(const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_kpe,
                           const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qp,
                           const AttnParams prm) {
    using C = AttnCfg<HG>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* pair_base = smem + C::kOffPair;
    uint8_t* kpe_base = smem + C::kOffKpe;
    uint8_t* q_base = smem + C::kOffQ;
    uint8_t* p_base = smem + C::kOffP;
    AttnMisc* misc = reinterpret_cast<AttnMisc*>(smem + C::kOffMisc);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int unit = blockIdx.x / prm.head_groups;
    const int group = blockIdx.x % prm.head_groups;
    const int seg_begin = prm.unit_ptr[unit];
    const int seg_end = prm.unit_ptr[unit + 1];
    const int P = prm.page_size;

    if (threadIdx.x == 0) {
        MLA_TRACE_CTA(0);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&misc->q_full[i], 1);
            mbar_init(&misc->q_empty[i], 1);
            mbar_init(&misc->s_full[i], 1);
            mbar_init(&misc->p_full[i], C::kSoftmaxThreads / 32);   // one arrival per softmax warp
        }
        mbar_init(&misc->pv_done, 1);
        mbar_init(&misc->o_full, 1);
        mbar_init(&misc->drain, 1);
        for (int i = 0; i < C::kKpeSlots; ++i) {
            mbar_init(&misc->kfull[i], 1);
            mbar_init(&misc->kempty[i], 1);
        }
        for (int i = 0; i < C::kPairSlots; ++i) {
            mbar_init(&misc->pfull[i], 1);
            mbar_init(&misc->pempty[i], 1);
            mbar_init(&misc->pload[i], 1);
        }
        misc->abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&misc->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tm_ckv);
            prefetch_tensormap(&tm_kpe);
            prefetch_tensormap(&tm_qn);
            prefetch_tensormap(&tm_qp);
        }
        uint32_t kcount = 0, pcount = 0, nq = 0;
        uint32_t pload_uses[C::kPairSlots];
#pragma unroll
        for (int i = 0; i < C::kPairSlots; ++i) pload_uses[i] = 0;
        bool ok = true;
        TileCursor cur;
        bool more = cur.init(prm.segments, seg_begin, seg_end);
        bool new_seg = true;
        int win_base = -(1 << 30), win_page = 0;
        const int32_t* pages = nullptr;
        uint32_t tile_idx = 0;
        // L2 prefetch cursor, kPrefetchTiles tiles ahead of the loads
        TileCursor pf;
        bool pf_more = pf.init(prm.segments, seg_begin, seg_end);
        bool pf_new = true;
        int pf_win_base = -(1 << 30), pf_win_page = 0;
        const int32_t* pf_pages = nullptr;
        auto prefetch_next_tile = [&]() {
            if (!pf_more) return;
            if (pf_new) {
                pf_pages = prm.kv_indices + prm.kv_indptr[pf.sg.b];
                pf_win_base = -(1 << 30);
            }
            const int fp = pf.t0 / P;
            const int np = (pf.ntok() + P - 1) / P;
            if (fp + np > pf_win_base + 32) {
                const int last_page = (pf.sg.t_end - 1) / P;
                pf_win_base = fp;
                pf_win_page = (pf_win_base + lane <= last_page) ? pf_pages[pf_win_base + lane] : 0;
            }
            const int pg = __shfl_sync(0xffffffffu, pf_win_page, (fp - pf_win_base + lane) & 31);
            if (lane < np) {
                l2_prefetch(prm.ckv + static_cast<size_t>(pg) * P * (kDimCkv * 2), static_cast<uint32_t>(P * kDimCkv * 2));
                l2_prefetch(prm.kpe + static_cast<size_t>(pg) * P * (kDimKpe * 2), static_cast<uint32_t>(P * kDimKpe * 2));
            }
            pf_more = pf.advance(pf_new);
        };
        for (int d = 0; d < C::kPrefetchTiles; ++d) prefetch_next_tile();
        while (more && ok) {
            prefetch_next_tile();
            if (new_seg) {
                pages = prm.kv_indices + prm.kv_indptr[cur.sg.b];
                win_base = -(1 << 30);
                const uint32_t qb = nq % C::kQBufs, use = nq / C::kQBufs;
                if (lane == 0) {
                    if (use > 0) ok = wait_phase(&misc->q_empty[qb], (use - 1) & 1, misc, prm.status, 1);
                    if (ok) {
                        uint8_t* q = q_base + qb * C::kQStride;
                        mbar_arrive_expect_tx(&misc->q_full[qb], C::kQBytes);
                        const int row = cur.sg.b * prm.h_q + group * HG;
                        for (int c = 0; c < 8; ++c)
                            tma_load_2d(q + c * C::kQChunkBytes, &tm_qn, &misc->q_full[qb], c * 64, row);
                        tma_load_2d(q + 8 * C::kQChunkBytes, &tm_qp, &misc->q_full[qb], 0, row);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                ++nq;
                if (!ok) break;
            }
            const int ntok = cur.ntok();
            const int first_page = cur.t0 / P;
            const int npages = (ntok + P - 1) / P;
            if (first_page + npages > win_base + 32) {  // refill the 32-page index window
                const int seg_last_page = (cur.sg.t_end - 1) / P;
                win_base = first_page;
                win_page = (win_base + lane <= seg_last_page) ? pages[win_base + lane] : 0;
            }
            const uint32_t bytes = static_cast<uint32_t>(npages * P * 128);
            // kpe rows of the tile
            {
                const uint32_t s = kcount % C::kKpeSlots, use = kcount / C::kKpeSlots;
                if (lane == 0 && use > 0) ok = wait_phase(&misc->kempty[s], (use - 1) & 1, misc, prm.status, 2);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                if (lane == 0) mbar_arrive_expect_tx(&misc->kfull[s], bytes);
                uint8_t* dst = kpe_base + s * C::kChunkBytes;
                for (int i = 0; i < npages; ++i) {
                    const int pg = __shfl_sync(0xffffffffu, win_page, first_page - win_base + i);
                    if (lane == 0) tma_load_2d(dst + i * P * 128, &tm_kpe, &misc->kfull[s], 0, pg * P);
                }
                if (lane == 0) MLA_TRACE_EVENT(0, tile_idx);
                ++kcount;
            }
            // ckv rows, one pair slot per 128 latent dims
            const bool partial = ntok < kTileTokens;
            for (int c = 0; c < 4 && ok; ++c) {
                const uint32_t s = pcount % C::kPairSlots, use = pcount / C::kPairSlots;
                if (lane == 0 && use > 0) ok = wait_phase(&misc->pempty[s], (use - 1) & 1, misc, prm.status, 3);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                uint64_t* bar = partial ? &misc->pload[s] : &misc->pfull[s];
                if (lane == 0) mbar_arrive_expect_tx(bar, 2 * bytes);
                uint8_t* dst = pair_base + s * C::kPairBytes;
                for (int i = 0; i < npages; ++i) {
                    const int pg = __shfl_sync(0xffffffffu, win_page, first_page - win_base + i);
                    if (lane == 0) {
                        tma_load_2d(dst + i * P * 128, &tm_ckv, bar, (2 * c) * 64, pg * P);
                        tma_load_2d(dst + C::kChunkBytes + i * P * 128, &tm_ckv, bar, (2 * c + 1) * 64, pg * P);
                    }
                }
                if (partial) {
                    // rows past the request's last token may hold stale or NaN bytes: zero them before
                    // publishing (a zero key row only changes scores that the softmax masks anyway)
                    if (lane == 0) ok = wait_phase(&misc->pload[s], pload_uses[s] & 1, misc, prm.status, 11);
                    ++pload_uses[s];
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    for (int r = ntok + lane; r < kTileTokens; r += 32) {
                        uint4* r0 = reinterpret_cast<uint4*>(dst + r * 128);
                        uint4* r1 = reinterpret_cast<uint4*>(dst + C::kChunkBytes + r * 128);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            r0[i] = make_uint4(0, 0, 0, 0);
                            r1[i] = make_uint4(0, 0, 0, 0);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&misc->pfull[s]);
                }
                if (lane == 0 && c == 3) MLA_TRACE_EVENT(1, tile_idx);
                ++pcount;
            }
            ++tile_idx;
            more = cur.advance(new_seg);
        }
        // teardown: let every copy this warp issued land before the CTA can exit
        if (lane == 0) {
            MLA_TRACE_CTA(1);
            const uint64_t t0 = global_timer_ns();
            auto drain = [&](uint64_t* bar, uint32_t uses) {
                if (uses == 0) return;
                while (!mbar_try_wait(bar, (uses - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
            };
            for (int b = 0; b < C::kQBufs; ++b)
                drain(&misc->q_full[b], nq / C::kQBufs + (static_cast<uint32_t>(b) < nq % C::kQBufs ? 1 : 0));
            for (int s = 0; s < C::kKpeSlots; ++s)
                drain(&misc->kfull[s], kcount / C::kKpeSlots + (static_cast<uint32_t>(s) < kcount % C::kKpeSlots ? 1 : 0));
            for (int s = 0; s < C::kPairSlots; ++s) {
                drain(&misc->pfull[s], pcount / C::kPairSlots + (static_cast<uint32_t>(s) < pcount % C::kPairSlots ? 1 : 0));
                drain(&misc->pload[s], pload_uses[s]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // base descriptors; per-MMA descriptors add (byte offset >> 4) to them
            const uint64_t qdesc0 = umma_desc_sw128_c<16, 1024>(smem_u32(q_base));      // Q^T, K-major
            const uint64_t pdesc0 = umma_desc_sw128_c<16, 1024>(smem_u32(p_base));      // P^T, K-major
            const uint64_t kdesc0 = umma_desc_sw128_c<16, 1024>(smem_u32(kpe_base));    // kpe rows, K-major
            const uint64_t sdesc0 = umma_desc_sw128_c<16, 1024>(smem_u32(pair_base));   // ckv rows, K-major
            const uint64_t vdesc0 =                                                     // ckv rows as V^T, MN-major
                umma_desc_sw128_c<C::kChunkBytes, 1024>(smem_u32(pair_base));
            // score side: tile s_tile, next block s_blk (0 = kpe, 1..4 = ckv pair s_blk - 1)
            TileCursor sc;
            bool s_more = sc.init(prm.segments, seg_begin, seg_end);
            uint32_t s_tile = 0, s_blk = 0, kcount = 0, s_pcount = 0, nq = 0;
            bool q_ready = false;
            // PV side: tile pv_tile, next 128-dim block pv_blk (its pair slot was filled for the score)
            TileCursor pc;
            bool pv_more = pc.init(prm.segments, seg_begin, seg_end);
            uint32_t pv_tile = 0, pv_blk = 0, pv_pcount = 0;
            bool p_ready = false;
            uint64_t idle_since = global_timer_ns();
            while (s_more || pv_more) {
                bool progressed = false;
                // ---- next PV block: needs S(pv_tile) issued and P(pv_tile) written; frees a pair slot
                if (pv_more && pv_tile < s_tile) {
                    if (!p_ready) p_ready = mbar_test_wait(&misc->p_full[pv_tile & 1], (pv_tile >> 1) & 1);
                    if (p_ready) {
                        tc_fence_after();
                        const uint32_t ps = pv_pcount % C::kPairSlots;
                        const uint64_t da = vdesc0 + ps * (C::kPairBytes >> 4);
                        const uint64_t db = pdesc0 + (pv_tile % C::kPBufs) * (C::kPStride >> 4);
                        const uint32_t d = tmem + C::kTmemO + pv_blk * HG;
                        const bool init = pc.first();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_bf16(d, da + kk * (2048 >> 4),
                                      db + (kk >> 2) * (C::kPChunkBytes >> 4) + (kk & 3) * (32 >> 4), C::kIdescPV,
                                      (init && kk == 0) ? 0u : 1u);
                        umma_commit(&misc->pempty[ps]);
                        ++pv_pcount;
                        if (++pv_blk == 4) {
                            umma_commit(&misc->pv_done);
                            if (pc.last()) umma_commit(&misc->o_full);
                            MLA_TRACE_EVENT(6, pv_tile);
                            ++pv_tile;
                            pv_blk = 0;
                            p_ready = false;
                            bool new_seg;
                            pv_more = pc.advance(new_seg);
                        }
                        progressed = true;
                    }
                }
                // ---- next score block: S(s_tile) may start once PV(s_tile - 2) is fully issued
                if (s_more && s_tile <= pv_tile + 1) {
                    const uint32_t qb = nq % C::kQBufs;
                    if (!q_ready) q_ready = mbar_test_wait(&misc->q_full[qb], (nq / C::kQBufs) & 1);
                    const uint64_t dq = qdesc0 + qb * (C::kQStride >> 4);
                    const uint32_t d = tmem + (s_tile & 1) * HG;
                    if (q_ready && s_blk == 0) {
                        const uint32_t ks = kcount % C::kKpeSlots;
                        if (mbar_test_wait(&misc->kfull[ks], (kcount / C::kKpeSlots) & 1)) {
                            tc_fence_after();
                            MLA_TRACE_EVENT(2, s_tile);
                            const uint64_t da = kdesc0 + ks * (C::kChunkBytes >> 4);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                umma_bf16(d, da + k * (32 >> 4), dq + 8 * (C::kQChunkBytes >> 4) + k * (32 >> 4),
                                          C::kIdescS, k > 0 ? 1u : 0u);
                            umma_commit(&misc->kempty[ks]);
                            ++kcount;
                            s_blk = 1;
                            progressed = true;
                        }
                    } else if (q_ready) {
                        const uint32_t ps = s_pcount % C::kPairSlots;
                        if (mbar_test_wait(&misc->pfull[ps], (s_pcount / C::kPairSlots) & 1)) {
                            tc_fence_after();
                            const uint32_t c = s_blk - 1;
                            const uint64_t da = sdesc0 + ps * (C::kPairBytes >> 4);
                            const uint64_t db = dq + (2 * c) * (C::kQChunkBytes >> 4);
#pragma unroll
                            for (int h = 0; h < 2; ++h)
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    umma_bf16(d, da + h * (C::kChunkBytes >> 4) + k * (32 >> 4),
                                              db + h * (C::kQChunkBytes >> 4) + k * (32 >> 4), C::kIdescS, 1u);
                            ++s_pcount;
                            if (++s_blk == 5) {
                                if (sc.last()) umma_commit(&misc->q_empty[qb]);
                                umma_commit(&misc->s_full[s_tile & 1]);
                                MLA_TRACE_EVENT(3, s_tile);
                                ++s_tile;
                                s_blk = 0;
                                bool new_seg;
                                s_more = sc.advance(new_seg);
                                if (new_seg) {
                                    ++nq;
                                    q_ready = false;
                                }
                            }
                            progressed = true;
                        }
                    }
                }
                if (progressed) {
                    idle_since = global_timer_ns();
                } else {
                    if (*reinterpret_cast<volatile int*>(&misc->abort_flag)) break;
                    if (global_timer_ns() - idle_since > kWaitLimitNs) {
                        *reinterpret_cast<volatile int*>(&misc->abort_flag) = 1;
                        atomicCAS(prm.status, 0u, kStatusTimeout | 4u);
                        break;
                    }
                }
            }
            // teardown: every MMA issued by this thread completes before TMEM is freed
            umma_commit(&misc->drain);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&misc->drain, 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int sp = warp & 3;                 // TMEM sub-partition this warp may access
        const int row = sp * 32 + lane;          // TMEM lane: token of the tile / latent dim of O^T
        const int gtid = threadIdx.x - 64;       // 0..127 within the group
        uint32_t tcount = 0, nseg = 0;
        bool ok = true;
        for (int si = seg_begin; si < seg_end && ok; ++si) {
            const Segment sg = prm.segments[si];
            const size_t head0 = static_cast<size_t>(group) * HG;
            if (sg.t_end <= sg.t_begin) {
                // request with no tokens
                float* o = prm.out + (static_cast<size_t>(sg.b) * prm.h_q + head0) * kDimCkv;
                for (int i = gtid; i < HG * kDimCkv; i += C::kSoftmaxThreads) o[i] = 0.f;
                if (gtid < HG) prm.lse[static_cast<size_t>(sg.b) * prm.h_q + head0 + gtid] = -INFINITY;
                continue;
            }
            float m_run[HG], l_part[HG];
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                m_run[h] = -INFINITY;
                l_part[h] = 0.f;
            }
            for (int t0 = sg.t_begin; t0 < sg.t_end; t0 += kTileTokens, ++tcount) {
                const bool first_tile = (t0 == sg.t_begin);
                const int ntok = min(kTileTokens, sg.t_end - t0);
                const bool valid = row < ntok;
                ok = wait_phase(&misc->s_full[tcount & 1], (tcount >> 1) & 1, misc, prm.status, 8);
                const bool bad = named_barrier_or(1, C::kSoftmaxThreads,
                                                  !ok || *reinterpret_cast<volatile int*>(&misc->abort_flag));
                if (bad) { ok = false; break; }
                if (gtid == 0) MLA_TRACE_EVENT(4, tcount);
                tc_fence_after();
                float x[HG];
#pragma unroll
                for (int j = 0; j < HG / 16; ++j)
                    tmem_ld16(tmem_addr(tmem, sp * 32, (tcount & 1) * HG + 16 * j), x + 16 * j);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < HG; ++h) x[h] = valid ? x[h] * prm.scale_log2 : -INFINITY;
                // tile max per head over the 128 tokens
                float (*red)[32] = misc->red_max[tcount & 1];
#pragma unroll
                for (int h = 0; h < HG; ++h) {
                    const float m = warp_max(x[h]);
                    if (lane == 0) red[sp][h] = m;
                }
                named_barrier_sync(1, C::kSoftmaxThreads);
                bool rescale = false;
                float alpha[HG];
#pragma unroll
                for (int h = 0; h < HG; ++h) {
                    const float mt = fmaxf(fmaxf(red[0][h], red[1][h]), fmaxf(red[2][h], red[3][h]));
                    alpha[h] = 1.f;
                    if (mt > m_run[h] + 8.f) {
                        alpha[h] = exp2f(m_run[h] - mt);
                        m_run[h] = mt;
                        rescale = true;
                    }
                    l_part[h] *= alpha[h];
                }
                // The PV of the previous tile must have completed before O^T is rescaled, and (with a
                // single P buffer) before P is overwritten.
                if ((C::kPBufs == 1 && tcount > 0) || (rescale && !first_tile)) {
                    ok = wait_phase(&misc->pv_done, (tcount - 1) & 1, misc, prm.status, 10);
                    const bool bad2 = named_barrier_or(1, C::kSoftmaxThreads,
                                                       !ok || *reinterpret_cast<volatile int*>(&misc->abort_flag));
                    if (bad2) { ok = false; break; }
                    tc_fence_after();
                }
                if (rescale && !first_tile) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int j = 0; j < HG / 16; ++j) {
                            float o[16];
                            const uint32_t a = tmem_addr(tmem, sp * 32, C::kTmemO + c * HG + 16 * j);
                            tmem_ld16(a, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) o[i] *= alpha[16 * j + i];
                            tmem_st16(a, o);
                        }
                    }
                    tmem_wait_st();
                }
                // P^T[h][t] in bf16: K-major 128B-swizzled rows, 64 tokens per chunk
                {
                    uint8_t* pchunk = p_base + (tcount % C::kPBufs) * C::kPStride + (row >> 6) * C::kPChunkBytes;
                    const int col = row & 63;
#pragma unroll
                    for (int h = 0; h < HG; ++h) {
                        const float p = exp2f(x[h] - m_run[h]);
                        l_part[h] += p;
                        *reinterpret_cast<__nv_bfloat16*>(pchunk + sw128_offset(h, col)) = __float2bfloat16_rn(p);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&misc->p_full[tcount & 1]);
                if (gtid == 0) MLA_TRACE_EVENT(5, tcount);
            }
            if (!ok) break;
            // ---- epilogue: wait for the last PV, normalise, store
            ok = wait_phase(&misc->o_full, nseg & 1, misc, prm.status, 9);
            ++nseg;
            const bool bad = named_barrier_or(1, C::kSoftmaxThreads,
                                              !ok || *reinterpret_cast<volatile int*>(&misc->abort_flag));
            if (bad) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const float s = warp_sum(l_part[h]);
                if (lane == 0) misc->red_sum[sp][h] = s;
            }
            named_barrier_sync(1, C::kSoftmaxThreads);
            float inv_l[HG];
#pragma unroll
            for (int h = 0; h < HG; ++h)
                inv_l[h] = 1.f / ((misc->red_sum[0][h] + misc->red_sum[1][h]) + (misc->red_sum[2][h] + misc->red_sum[3][h]));
            float* obase;
            float* lbase;
            if (sg.slot < 0) {
                obase = prm.out + (static_cast<size_t>(sg.b) * prm.h_q + head0) * kDimCkv;
                lbase = prm.lse + static_cast<size_t>(sg.b) * prm.h_q + head0;
            } else {
                obase = prm.part_o + (static_cast<size_t>(sg.slot) * prm.h_q + head0) * kDimCkv;
                lbase = prm.part_lse + static_cast<size_t>(sg.slot) * prm.h_q + head0;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int j = 0; j < HG / 16; ++j) {
                    float o[16];
                    tmem_ld16(tmem_addr(tmem, sp * 32, C::kTmemO + c * HG + 16 * j), o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        obase[static_cast<size_t>(16 * j + i) * kDimCkv + c * 128 + row] = o[i] * inv_l[16 * j + i];
                }
            }
            if (gtid < HG) {
                float l = 0.f, m = 0.f;
#pragma unroll
                for (int h = 0; h < HG; ++h)
                    if (h == gtid) {
                        l = (misc->red_sum[0][h] + misc->red_sum[1][h]) + (misc->red_sum[2][h] + misc->red_sum[3][h]);
                        m = m_run[h];
                    }
                lbase[gtid] = (m + log2f(l)) * 0.69314718055994530942f;
            }
            tc_fence_before();
            if (sg.slot >= 0) {
                // ---- split request: the last piece to arrive merges all of them in slot order
                __threadfence();
                named_barrier_sync(1, C::kSoftmaxThreads);
                if (gtid == 0) {
                    const int old = atomicAdd(&prm.counters[sg.item * prm.head_groups + group], 1);
                    misc->merge_flag = (old == sg.n_slots - 1);
                }
                named_barrier_sync(1, C::kSoftmaxThreads);
                if (misc->merge_flag) {
                    if (gtid == 0) MLA_TRACE_CTA(4);
                    __threadfence();
                    merge_split_pieces<HG, C::kSoftmaxThreads>(prm, sg.b, sg.slot_begin, sg.n_slots, head0, gtid, 1,
                                                               misc->mrg_max, misc->mrg_inv, misc->mrg_w);
                    if (gtid == 0) prm.counters[sg.item * prm.head_groups + group] = 0;
                    if (gtid == 0) MLA_TRACE_CTA(5);
                }
            }
            // red_sum / merge scratch are reused by the next segment only after this barrier
            named_barrier_sync(1, C::kSoftmaxThreads);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
    if (threadIdx.x == 0) MLA_TRACE_CTA(6);
}

}  // namespace mla
