// MLA paged decode attention for 128 query heads on sm_103a: a cluster of two CTAs per
// work unit, tcgen05 MMAs with M = 128 heads.
//
// Absorbed MLA decode is MQA with one KV head: key [ckv | kpe] (576), value ckv (512)
// ("Benchmarking MLA", FlashInfer issue #700).  With the heads on the MMA's M axis every
// softmax row is one TMEM lane, so each softmax thread owns one head and needs no
// cross-thread reduction -- but S (128 heads x 128 tokens fp32) and O (128 heads x 512
// dims fp32) together need 640 TMEM columns and an SM has 512.  The two CTAs of a cluster
// therefore split the work by role:
//
//   rank 0 ("S CTA"):  q_nope sits in TMEM (256 columns, the A operand), q_pe in shared
//     memory; S = Q K^T is accumulated into one of two 128-column TMEM buffers by
//     36 MMAs (M 128, N 128, K 16) per 128-token tile from a ring of three K slots (latent
//     chunks 0-3 and 4-7, 64 KB each, then the rope part), filled with 4-D page boxes.
//     The softmax warpgroup (thread = head) reads S, keeps the running max and sum, and
//     writes P (bf16) and the rescale factors into a local staging tile, which one thread
//     hands to rank 1's shared memory with bulk copies (cp.async.bulk over the cluster).
//     Per-thread remote stores of P (st.shared::cluster) measured 17 % slower per step:
//     thousands of 16-byte transactions per tile held up the SM's TMA loads.
//   rank 1 ("O CTA"):  O (128 x 512 fp32) fills its TMEM; O += P V is 16 MMAs (M 128,
//     N 256, K 16) per tile, V streamed in 64-token slots of 256 dims through the same 4-D
//     page view as the keys.  A correction
//     warpgroup rescales O rows when rank 0 raised a head's running max (lazily, by more
//     than 2^8), zeroes value rows past the last token of a partial tile, and writes the
//     normalised output (or a split piece's partial) at the end of a segment.
//
// 64-head requests run on the same kernel with the MMAs' M padded to 128: heads 64..127
// get zero query rows and zero P rows, and nothing is written for them.
//
// The split-KV partition, the partials and the last-arriver merge are those of the other
// kernels (FlashMLA PR #233, "balanced scheduler, deterministic combine").  Every wait is
// bounded; a wait that runs out raises the abort flag of both CTAs.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace mla {

struct PairCfg {
    static constexpr int kThreads = 256;          // 8 warps: producers (0, 2, 3), MMA (1), one warpgroup (4-7)
    // Copy issue: one issuing thread starts about one ring slot per ~0.45 us (measured on this GPU,
    // whatever the box shape, from HBM or L2), so each CTA spreads its copies over three
    // producer warps.  Producer p owns the ring slots s with s % (producers) == p, so every slot
    // has one issuer and each producer can drain its own slots on its own.
    static constexpr int kKProducers = 3;         // rank 0: warps 0, 2, 3
    static constexpr int kVProducers = 2;         // rank 1: warps 0, 2
    static constexpr int kTile = kTileTokens;     // 128 tokens
    static constexpr int kChunkBytes = 128 * 128; // 128 rows x 128 B (64 bf16)
    // rank 0
    // K of a tile in 3 slots, one per producer: chunks 0-3 and 4-7 of the latent (64 KB each, one
    // 4-D box of 4 chunks per page: [row group][chunk][8 rows][128 B], 8-row groups 4 KB apart),
    // then the rope chunk (16 KB, one 2-D box per page).  Large boxes: one SM's copy engine moves
    // ~1.5x the bytes per microsecond of 8 KB boxes for the same bytes in flight (measured).
    static constexpr int kKSlots = 3;
    static constexpr int kKSlotBytes = 4 * kChunkBytes;   // latent slots; the rope slot uses kChunkBytes
    // A P buffer: the P tile [2 token chunks][128 heads][128 B], then the tile's per-head factors
    // (PairHand); rank 0 stages one and hands it to rank 1 with a single bulk copy.
    static constexpr int kPTileBytes = 2 * kChunkBytes;
    static constexpr int kPBufBytes = kPTileBytes + 2048;              // 1024-aligned stride
    static constexpr int kOffQpe = 0;                                  // [128 heads][128 B] SW128
    static constexpr int kOffK = kOffQpe + kChunkBytes;                // K ring
    static constexpr int kOffPStage = kOffK + 9 * kChunkBytes;         // P of one tile, copied to rank 1
    static constexpr int kSEnd = kOffPStage + kPBufBytes;              // 194 KB
    // rank 1
    static constexpr int kPBufs = 2;
    static constexpr int kOffP = 0;
    // a V slot: 64 tokens x 256 dims as [row group][4 chunks][8 rows][128 B] (4-D page boxes, the
    // MN-major value operand: 64-dim groups 1 KB apart, 8-token groups 4 KB apart)
    static constexpr int kVSlotBytes = 64 * 4 * 128;
    static constexpr int kVSlots = 4;             // a whole tile's values; producer = slot % 2
    static constexpr int kOffV = kOffP + kPBufs * kPBufBytes;
    static constexpr int kOEnd = kOffV + kVSlots * kVSlotBytes;        // 196 KB
    static constexpr int kOffMisc = kSEnd > kOEnd ? kSEnd : kOEnd;
    static constexpr int kMiscBytes = 12 * 1024;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static constexpr uint32_t kTmemQ = 0;      // rank 0: q_nope, 256 columns
    static constexpr uint32_t kTmemS = 256;    // rank 0: S buffers at 256, 384
    static constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16(128, 256, false, true);
    static_assert(kKSlots % kKProducers == 0 && kVSlots % kVProducers == 0, "each slot has one producer");
};

// Per-head factors of one tile, handed to rank 1 right after the tile's P in the same buffer.
struct PairHand {
    float alpha[128];   // the rescale factor for each head (1 if its running max did not move)
    float fin_m[128];   // at a segment's last tile: running max (log2 units)
    float fin_l[128];   // ... and row sum
    int rescale[4];     // [0]: some head's running max moved
};
static_assert(PairCfg::kPTileBytes + sizeof(PairHand) <= PairCfg::kPBufBytes, "P buffer layout");
constexpr uint32_t kPairHandBytes = PairCfg::kPTileBytes + sizeof(PairHand);   // one bulk copy per tile
static_assert(kPairHandBytes % 16 == 0, "bulk copy size");

__device__ __forceinline__ PairHand* pair_hand(uint8_t* pbuf) {
    return reinterpret_cast<PairHand*>(pbuf + PairCfg::kPTileBytes);
}

// Producer index of a warp of the two-CTA kernel (warps 0, 2, 3), or -1.
__device__ __forceinline__ int pair_producer(int warp) { return warp == 0 ? 0 : (warp == 2 || warp == 3 ? warp - 1 : -1); }

// Same layout in both CTAs, so mapa_shared of a field's address reaches the partner's copy.
struct PairMisc {
    // rank 0
    uint64_t k_full[PairCfg::kKSlots], k_empty[PairCfg::kKSlots];
    uint64_t s_full[2], s_empty[2];
    uint64_t q_full, q_empty;
    uint64_t p_empty[PairCfg::kPBufs];
    // rank 1
    uint64_t v_full[PairCfg::kVSlots], v_empty[PairCfg::kVSlots];
    uint64_t p_full[PairCfg::kPBufs];
    uint64_t pv_done[PairCfg::kPBufs];
    // Zeroing the value rows past the last token of a partial tile, per half: the MMA thread
    // (the V ring's consumer) raises vz_go once the slot has landed, the correction warps zero
    // the rows and raise vz_done.  One barrier pair per half, so that no barrier can run two
    // phases ahead of its waiter.
    uint64_t corr_done, vz_go[2], vz_done[2], epi_done;
    uint32_t tmem_base;
    int abort_flag;
    int merge_flag;
    float mrg_max[128], mrg_inv[128], mrg_w[8 * 128];
};

// Debug builds (-DMLA_TRACE): each role's progress counter, readable by the host while the
// kernel runs when the trace buffer is mapped host memory.
#ifdef MLA_TRACE
#define PAIR_PROGRESS(k, v)                                                                                    \
    do {                                                                                                      \
        if (prm.trace)                                                                                        \
            reinterpret_cast<volatile uint64_t*>(prm.trace)[4 * 8 * 256 + blockIdx.x * 8 + (k)] = (uint64_t)(v); \
    } while (0)
#else
#define PAIR_PROGRESS(k, v) \
    do {                    \
    } while (0)
#endif

// Bounded wait on a local mbarrier phase.  kCluster: the phase is completed by arrivals from
// the partner CTA, whose writes the wait acquires (cluster scope); otherwise by this CTA's
// threads, its TMA copies or its tensor-core commits (CTA scope).  On a timeout it raises both
// CTAs' abort flags and records `site`.
template <bool kCluster = false>
__device__ __forceinline__ bool pair_wait(uint64_t* bar, uint32_t parity, PairMisc* misc, uint32_t partner_abort,
                                          uint32_t* status, uint32_t site) {
    auto probe = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (probe()) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (probe()) return true;
        if (*reinterpret_cast<volatile int*>(&misc->abort_flag)) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *reinterpret_cast<volatile int*>(&misc->abort_flag) = 1;
            st_cluster_u32(partner_abort, 1u);
            atomicCAS(status, 0u, kStatusTimeout | site);
            return false;
        }
    }
}

// HQ: query heads, 128, or 64 with the MMAs' M padded to 128.  F16: IEEE fp16 q, ckv and kpe
// (and P) instead of bf16; the MMAs take the matching operand format.
template <int HQ, bool F16 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg::kThreads, 1)
    mla_decode_pair_kernel(const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_kpe,
                           const __grid_constant__ CUtensorMap tm_qpe, const __grid_constant__ CUtensorMap tm_v,
                           const AttnParams prm, const uint16_t* __restrict__ q_nope) {
    using C = PairCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PairMisc* misc = reinterpret_cast<PairMisc*>(smem + C::kOffMisc);
    static_assert(sizeof(PairMisc) <= C::kMiscBytes, "misc region");

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const uint32_t partner = rank ^ 1u;
    const int unit = blockIdx.x / 2;
    const int seg_begin = prm.unit_ptr[unit];
    const int seg_end = prm.unit_ptr[unit + 1];
    const int P = prm.page_size;
    static_assert(HQ == 64 || HQ == 128, "the two-CTA kernel serves 64 or 128 heads");
    constexpr uint32_t kIdS = F16 ? idesc_f16(128, 128, false, false) : C::kIdescS;
    constexpr uint32_t kIdPV = F16 ? idesc_f16(128, 256, false, true) : C::kIdescPV;
    constexpr int hq = HQ;
    const uint32_t partner_abort = mapa_shared(smem_u32(&misc->abort_flag), partner);

    // Prologue before the previous kernel in the stream has finished (programmatic dependent
    // launch): barriers, TMEM and this unit's slice of the plan, which only the plan commit
    // writes.  Every read of the caller's buffers and every write comes after grid_dep_wait.
    grid_dep_launch();
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kKSlots; ++i) {
            mbar_init(&misc->k_full[i], 1);
            mbar_init(&misc->k_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&misc->s_full[i], 1);
            mbar_init(&misc->s_empty[i], 4);
        }
        for (int i = 0; i < C::kPBufs; ++i) {
            mbar_init(&misc->p_empty[i], 1);
            mbar_init(&misc->p_full[i], 1);   // rank 0's issuing thread; the copies add bytes
            mbar_init(&misc->pv_done[i], 1);
        }
        mbar_init(&misc->q_full, 2);
        mbar_init(&misc->q_empty, 1);
        for (int i = 0; i < C::kVSlots; ++i) {
            mbar_init(&misc->v_full[i], 1);
            mbar_init(&misc->v_empty[i], 1);
        }
        mbar_init(&misc->corr_done, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&misc->vz_go[i], 1);
            mbar_init(&misc->vz_done[i], 1);
        }
        mbar_init(&misc->epi_done, 1);
        misc->abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&misc->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers exist before any remote arrive
    grid_dep_wait();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&misc->abort_flag) != 0; };

    if (rank == 0) {
        // ================================================================== S CTA
        if (pair_producer(warp) >= 0) {
            // ---------------------------------------------------------- TMA producers: q_pe, K chunks
            // producer pid issues the chunks of slots s % kKProducers == pid (and q_pe if pid == 0)
            const int pid = pair_producer(warp);
            if (lane == 0) {
                prefetch_tensormap(&tm_ckv);
                prefetch_tensormap(&tm_kpe);
                prefetch_tensormap(&tm_qpe);
            }
            uint32_t kcount = 0, segc = 0;
            bool ok = true;
            TileCursorT<C::kTile> cur;
            bool more = cur.init(prm.segments, seg_begin, seg_end);
            bool new_seg = true;
            int win_base = -(1 << 30), win_page = 0;
            const int32_t* pages = nullptr;
            while (more && ok) {
                if (new_seg) {
                    if (pid == 0 && lane == 0 && segc > 0)
                        ok = pair_wait(&misc->q_empty, (segc - 1) & 1, misc, partner_abort, prm.status, 41);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    if (pid == 0 && lane == 0) {
                        mbar_arrive_expect_tx(&misc->q_full, 128 * 128);
                        // 128 rows from the request's first head: for 64 heads the rows past them
                        // belong to the next request (or lie past the tensor, filled with zeros) and
                        // only feed score rows that are never used
                        tma_load_2d(smem + C::kOffQpe, &tm_qpe, &misc->q_full, 0, cur.sg.b * hq);
                    }
                    ++segc;
                    pages = prm.kv_indices + prm.kv_indptr[cur.sg.kv];
                    win_base = -(1 << 30);
                }
                const int ntok = cur.ntok();
                const int nbox = (ntok + P - 1) / P;
                const int first_page = cur.t0 / P;
                if (first_page + nbox > win_base + 32 || first_page < win_base) {
                    const int seg_last_page = (cur.sg.t_end - 1) / P;
                    win_base = first_page;
                    win_page = (win_base + lane <= seg_last_page) ? pages[win_base + lane] : 0;
                }
                for (int sl = 0; sl < C::kKSlots && ok; ++sl) {   // latent chunks 0-3, 4-7, then kpe
                    const uint32_t s = kcount % C::kKSlots, use = kcount / C::kKSlots;
                    if (static_cast<int>(s) % C::kKProducers != pid) {   // another producer's slot
                        ++kcount;
                        continue;
                    }
                    if (lane == 0 && sl == 2) MLA_TRACE_EVENT(0, kcount / C::kKSlots);
                    if (lane == 0 && use > 0)
                        ok = pair_wait(&misc->k_empty[s], (use - 1) & 1, misc, partner_abort, prm.status, 42);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    if (lane == 0) MLA_TRACE_UNIT(0, kcount);
                    uint8_t* dst = smem + C::kOffK + s * C::kKSlotBytes;
                    const uint32_t row_bytes = sl < 2 ? 4 * 128 : 128;   // bytes a token brings into the slot
                    if (lane == 0) mbar_arrive_expect_tx(&misc->k_full[s], static_cast<uint32_t>(nbox * P) * row_bytes);
                    for (int bx = 0; bx < nbox; ++bx) {
                        const int pg = __shfl_sync(0xffffffffu, win_page, (first_page + bx - win_base) & 31);
                        if (lane == 0) {
                            if (sl < 2)
                                tma_load_4d(dst + bx * P * row_bytes, &tm_ckv, &misc->k_full[s], 0, 0, 4 * sl,
                                            pg * (P / 8));
                            else
                                tma_load_2d(dst + bx * P * row_bytes, &tm_kpe, &misc->k_full[s], 0, pg * P);
                        }
                    }
                    if (lane == 0 && sl == 0) MLA_TRACE_EVENT(5, kcount / C::kKSlots);
                    if (lane == 0) MLA_TRACE_UNIT(1, kcount);
                    ++kcount;
                }
                if (pid == 0 && lane == 0) PAIR_PROGRESS(0, kcount);
                more = cur.advance(new_seg);
            }
            if (lane == 0) {   // let every copy of this producer's slots land before the CTA can exit
                const uint64_t t0 = global_timer_ns();
                for (int s = pid; s < C::kKSlots; s += C::kKProducers) {
                    const uint32_t uses = kcount / C::kKSlots + (static_cast<uint32_t>(s) < kcount % C::kKSlots ? 1 : 0);
                    if (uses == 0) continue;
                    while (!mbar_try_wait(&misc->k_full[s], (uses - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
                }
            }
        } else if (warp == 1) {
            // ---------------------------------------------------------- MMA issuer: S = Q K^T
            if (lane == 0) {
                uint32_t tcount = 0, kcount = 0, segc = 0;
                bool ok = true;
                TileCursorT<C::kTile> cur;
                bool more = cur.init(prm.segments, seg_begin, seg_end);
                bool new_seg = true;
                // descriptors of slot 0 / q_pe at k = 0; a slot or a 16-dim step only moves the start
                // address (in 16-byte units, no carry out of its field below 256 KB)
                // latent chunks: 8-row groups 4 KB apart (4 chunks of a row group side by side)
                const uint64_t kdesc0 = umma_desc_sw128_c<16, 4096>(smem_u32(smem + C::kOffK));
                const uint64_t rdesc0 = umma_desc_sw128_c<16, 1024>(smem_u32(smem + C::kOffK + 2 * C::kKSlotBytes));
                const uint64_t qdesc0 = umma_desc_sw128_c<16, 1024>(smem_u32(smem + C::kOffQpe));
                while (more && ok) {
                    const bool last = cur.last();
                    if (new_seg) {
                        ok = pair_wait(&misc->q_full, segc & 1, misc, partner_abort, prm.status, 43);
                        ++segc;
                    }
                    const uint32_t buf = tcount & 1, ub = tcount >> 1;
                    if (ok && ub > 0) ok = pair_wait(&misc->s_empty[buf], (ub - 1) & 1, misc, partner_abort, prm.status, 44);
                    if (!ok) break;
                    MLA_TRACE_EVENT(1, tcount);
                    tc_fence_after();
                    const uint32_t d = tmem + C::kTmemS + buf * 128;
                    // every tile fills each of the 3 slots once (chunks 0-3, 4-7, the rope chunk): a
                    // slot's use number is the tile count.  A slot is filled by TMA, so waiting on its
                    // barrier is enough to order the MMAs' reads after the copy (the tcgen05 fence
                    // above, once per tile, orders them after the softmax's reads of this S buffer).
                    static_assert(C::kKSlots == 3, "latent chunks 0-3, 4-7, then the rope chunk");
                    for (int c = 0; c < 9 && ok; ++c) {
                        const int sl = c < 8 ? c >> 2 : 2;
                        if ((c & 3) == 0) {   // first chunk of a slot: wait for it to land
                            ok = pair_wait(&misc->k_full[sl], tcount & 1, misc, partner_abort, prm.status, 45);
                            if (!ok) break;
                            MLA_TRACE_UNIT(2, kcount);
                        }
                        if (c < 8) {
                            const uint64_t bd = kdesc0 + static_cast<uint64_t>((sl * C::kKSlotBytes + (c & 3) * 1024) >> 4);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                umma_bf16_ts(d, tmem + C::kTmemQ + c * 32 + k * 8, bd + 2 * k, kIdS, (c | k) != 0);
                        } else {
#pragma unroll
                            for (int k = 0; k < 4; ++k) umma_bf16(d, qdesc0 + 2 * k, rdesc0 + 2 * k, kIdS, 1);
                        }
                        if ((c & 3) == 3 || c == 8) {   // last chunk of a slot: release it
                            umma_commit(&misc->k_empty[sl]);
                            MLA_TRACE_UNIT(3, kcount);
                            ++kcount;
                        }
                    }
                    if (!ok) break;
                    umma_commit(&misc->s_full[buf]);
                    if (last) umma_commit(&misc->q_empty);
                    MLA_TRACE_EVENT(2, tcount);
                    ++tcount;
                    PAIR_PROGRESS(1, tcount);
                    more = cur.advance(new_seg);
                }
            }
        } else if (warp >= 4) {
            // ---------------------------------------------------------- softmax warpgroup: thread = head
            const int h = threadIdx.x - 128;
            const uint32_t lane_base = static_cast<uint32_t>(warp - 4) * 32;
            const uint32_t o_p = mapa_shared(smem_u32(smem + C::kOffP), partner);
            const uint32_t o_pfull = mapa_shared(smem_u32(&misc->p_full[0]), partner);
            uint8_t* pstage = smem + C::kOffPStage;
            PairHand* stage_hand = pair_hand(pstage);
            const uint32_t pstage_row = smem_u32(pstage) + h * 128;
            uint32_t tcount = 0, segc = 0;
            bool ok = true;
            for (int si = seg_begin; si < seg_end && ok; ++si) {
                const Segment sg = prm.segments[si];
                if (sg.t_end <= sg.t_begin) continue;
                // q_nope row of head h -> TMEM columns [0, 256) of lane h, once the previous
                // segment's score MMAs are done with it
                if (segc > 0) ok = pair_wait(&misc->q_empty, (segc - 1) & 1, misc, partner_abort, prm.status, 46);
                ok = !named_barrier_or(1, 128, !ok);
                if (!ok) break;
                {
                    const uint4* qrow =
                        reinterpret_cast<const uint4*>(q_nope + (static_cast<size_t>(sg.b) * hq + h) * kDimCkv);
#pragma unroll 1
                    for (int c0 = 0; c0 < 256; c0 += 32) {
                        uint32_t r[32];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 v = h < hq ? qrow[c0 / 4 + j] : make_uint4(0, 0, 0, 0);
                            r[4 * j] = v.x;
                            r[4 * j + 1] = v.y;
                            r[4 * j + 2] = v.z;
                            r[4 * j + 3] = v.w;
                        }
                        tmem_st32(tmem_addr(tmem, lane_base, C::kTmemQ + c0), r);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                named_barrier_sync(1, 128);
                if (h == 0) mbar_arrive(&misc->q_full);
                ++segc;
                float m_run = -INFINITY, l = 0.f;
                bool first = true;
                for (int t0 = sg.t_begin; t0 < sg.t_end && ok; t0 += C::kTile) {
                    const int ntok = min(C::kTile, sg.t_end - t0);
                    const uint32_t buf = tcount & 1, ub = tcount >> 1;                  // S buffer
                    const uint32_t pb = tcount % C::kPBufs, up = tcount / C::kPBufs;   // P buffer
                    ok = pair_wait(&misc->s_full[buf], ub & 1, misc, partner_abort, prm.status, 47);
                    if (ok && up > 0) ok = pair_wait<true>(&misc->p_empty[pb], (up - 1) & 1, misc, partner_abort, prm.status, 48);
                    if (h == 0) bulk_wait_read_all();   // the previous tile's copies have left the staging
                    ok = !named_barrier_or(1, 128, !ok || aborted());
                    if (!ok) break;
                    if (h == 0) MLA_TRACE_EVENT(3, tcount);
                    tc_fence_after();
                    float s[128];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t r[32];
                        tmem_ld32(tmem_addr(tmem, lane_base, C::kTmemS + buf * 128 + 32 * j), r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) s[32 * j + i] = __uint_as_float(r[i]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&misc->s_empty[buf]);
                    if (h == 0) MLA_TRACE_EVENT(6, tcount);
                    float mt = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 128; ++i) {
                        if (i >= ntok || h >= hq) s[i] = -INFINITY;   // padded heads: P = 0
                        mt = fmaxf(mt, s[i]);
                    }
                    if (h >= hq) mt = 0.f;
                    // lazy running max (log2 units): move it only when the tile max exceeds it by 8
                    const float ms = mt * prm.scale_log2;
                    float alpha = 1.f;
                    bool resc = false;
                    if (ms > m_run + 8.f) {
                        alpha = first ? 0.f : exp2f(m_run - ms);
                        resc = !first;
                        m_run = ms;
                        l *= alpha;
                    }
                    // P row of head h -> the staging tile, K-major with the 128-byte swizzle
#pragma unroll
                    for (int ck = 0; ck < 2; ++ck) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int t = 64 * ck + 8 * u + 2 * e;
                                const float p0 = fast_exp2(fmaf(s[t], prm.scale_log2, -m_run));
                                const float p1 = fast_exp2(fmaf(s[t + 1], prm.scale_log2, -m_run));
                                l += p0 + p1;
                                if constexpr (F16) {
                                    __half2 v = __floats2half2_rn(p0, p1);
                                    w[e] = *reinterpret_cast<uint32_t*>(&v);
                                } else {
                                    __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
                                    w[e] = *reinterpret_cast<uint32_t*>(&v);
                                }
                            }
                            st_shared_v4(pstage_row + ck * C::kChunkBytes + ((u ^ (h & 7)) << 4), w[0], w[1], w[2], w[3]);
                        }
                    }
                    stage_hand->alpha[h] = alpha;
                    stage_hand->fin_m[h] = m_run;
                    stage_hand->fin_l[h] = l;
                    fence_proxy_async_smem();   // this thread's staging writes -> the copy engine
                    if (h == 0) MLA_TRACE_EVENT(7, tcount);
                    const bool any = named_barrier_or(2, 128, resc);
                    if (h == 0) {
                        stage_hand->rescale[0] = any ? 1 : 0;
                        fence_proxy_async_smem();
                        const uint32_t bar = o_pfull + pb * 8;
                        // P and the factors in one copy
                        mbar_arrive_expect_tx_cluster(bar, kPairHandBytes);
                        bulk_copy_to_cluster(o_p + pb * C::kPBufBytes, pstage, kPairHandBytes, bar);
                        bulk_commit_group();
                        MLA_TRACE_EVENT(4, tcount);
                    }
                    first = false;
                    ++tcount;
                    if (h == 0) PAIR_PROGRESS(2, tcount);
                }
            }
            if (h == 0) bulk_wait_read_all();
        }
    } else {
        // ================================================================== O CTA
        if (pair_producer(warp) >= 0 && pair_producer(warp) < C::kVProducers) {
            // ---------------------------------------------------------- TMA producers: V slots
            // producer pid issues the slots s % kVProducers == pid
            const int pid = pair_producer(warp);
            if (lane == 0) prefetch_tensormap(&tm_v);
            uint32_t vcount = 0;
            bool ok = true;
            TileCursorT<C::kTile> cur;
            bool more = cur.init(prm.segments, seg_begin, seg_end);
            bool new_seg = true;
            int win_base = -(1 << 30), win_page = 0;
            const int32_t* pages = nullptr;
            while (more && ok) {
                if (new_seg) {
                    pages = prm.kv_indices + prm.kv_indptr[cur.sg.kv];
                    win_base = -(1 << 30);
                }
                const int ntok = cur.ntok();
                const int nv = (ntok + 63) / 64;   // 64-token V slots per half
                const int first_page = cur.t0 / P;
                const int last_page = (cur.t0 + nv * 64 - 1) / P;
                if (last_page + 1 > win_base + 32 || first_page < win_base) {
                    const int seg_last_page = (cur.sg.t_end - 1) / P;
                    win_base = first_page;
                    win_page = (win_base + lane <= seg_last_page) ? pages[win_base + lane] : 0;
                }
                for (int half = 0; half < 2 && ok; ++half) {
                    for (int q = 0; q < nv && ok; ++q) {
                        const uint32_t s = vcount % C::kVSlots, use = vcount / C::kVSlots;
                        if (static_cast<int>(s) % C::kVProducers != pid) {   // another producer's slot
                            ++vcount;
                            continue;
                        }
                        if (lane == 0 && use > 0)
                            ok = pair_wait(&misc->v_empty[s], (use - 1) & 1, misc, partner_abort, prm.status, 51);
                        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                        if (!ok) break;
                        uint8_t* dst = smem + C::kOffV + s * C::kVSlotBytes;
                        if (lane == 0) MLA_TRACE_UNIT1(3, vcount);
                        if (lane == 0) mbar_arrive_expect_tx(&misc->v_full[s], C::kVSlotBytes);
                        if (pid == 0 && lane == 0 && half == 0 && q == 0) MLA_TRACE_EVENT(0, vcount / (2 * nv));
                        if (pid == 0 && lane == 0 && half == 1 && q == nv - 1) MLA_TRACE_EVENT(1, vcount / (2 * nv));
                        // whole pages (a slot starts on a page boundary); past the request's last page
                        // the page table window gives page 0, whose rows feed no MMA step
                        for (int bx = 0; bx < 64 / P; ++bx) {
                            const int t = cur.t0 + q * 64 + bx * P;
                            const int pg = __shfl_sync(0xffffffffu, win_page, (t / P - win_base) & 31);
                            if (lane == 0)
                                tma_load_4d(dst + bx * P * 512, &tm_v, &misc->v_full[s], 0, 0, 4 * half, pg * (P / 8));
                        }
                        ++vcount;
                    }
                }
                if (pid == 0 && lane == 0) PAIR_PROGRESS(3, vcount);
                more = cur.advance(new_seg);
            }
            if (lane == 0) {   // this producer's slots
                const uint64_t t0 = global_timer_ns();
                for (int s = pid; s < C::kVSlots; s += C::kVProducers) {
                    const uint32_t uses = vcount / C::kVSlots + (static_cast<uint32_t>(s) < vcount % C::kVSlots ? 1 : 0);
                    if (uses == 0) continue;
                    while (!mbar_try_wait(&misc->v_full[s], (uses - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
                }
            }
        } else if (warp == 1) {
            // ---------------------------------------------------------- MMA issuer: O += P V
            if (lane == 0) {
                uint32_t tcount = 0, vcount = 0, segc = 0, rcount = 0, zcount = 0;
                bool ok = true;
                TileCursorT<C::kTile> cur;
                bool more = cur.init(prm.segments, seg_begin, seg_end);
                bool new_seg = true;
                const uint64_t pdesc0 = umma_desc_sw128_c<16, 1024>(smem_u32(smem + C::kOffP));
                const uint64_t vdesc0 = umma_desc_sw128_c<1024, 4096>(smem_u32(smem + C::kOffV));
                while (more && ok) {
                    const bool first = cur.first();
                    const int ntok = cur.ntok();
                    const uint32_t buf = tcount % C::kPBufs, ub = tcount / C::kPBufs;
                    ok = pair_wait<true>(&misc->p_full[buf], ub & 1, misc, partner_abort, prm.status, 52);
                    if (ok && new_seg && segc > 0)
                        ok = pair_wait(&misc->epi_done, (segc - 1) & 1, misc, partner_abort, prm.status, 53);
                    if (new_seg) ++segc;
                    if (ok && !first && *reinterpret_cast<volatile int*>(&pair_hand(smem + C::kOffP + buf * C::kPBufBytes)->rescale[0])) {
                        ok = pair_wait(&misc->corr_done, rcount & 1, misc, partner_abort, prm.status, 54);
                        ++rcount;
                    }
                    if (!ok) break;
                    MLA_TRACE_EVENT(5, tcount);
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint64_t pdesc = pdesc0 + static_cast<uint64_t>((buf * C::kPBufBytes) >> 4);
                    const int nv = (ntok + 63) / 64;
                    const bool partial = (ntok & 15) != 0;
                    for (int half = 0; half < 2 && ok; ++half) {
                        for (int q = 0; q < nv && ok; ++q) {
                            const uint32_t s = vcount % C::kVSlots;
                            ok = pair_wait(&misc->v_full[s], (vcount / C::kVSlots) & 1, misc, partner_abort, prm.status, 56);
                            if (!ok) break;
                            MLA_TRACE_UNIT1(0, vcount);
                            if (partial && q == nv - 1) {
                                // the slot with the tile's last token: its rows past it are zeroed first
                                mbar_arrive(&misc->vz_go[half]);
                                ok = pair_wait(&misc->vz_done[half], zcount & 1, misc, partner_abort, prm.status, 55);
                                if (!ok) break;
                                fence_proxy_async_smem();
                                tc_fence_after();
                            }
                            // a TMA-filled slot: its barrier wait orders the MMAs' reads after the copy
                            const uint64_t bslot = vdesc0 + static_cast<uint64_t>((s * C::kVSlotBytes) >> 4);
                            for (int k4 = 0; k4 < 4; ++k4) {
                                const int kk = 4 * q + k4;   // 16-token step within the tile
                                if (16 * kk >= ntok) break;
                                const uint64_t ad = pdesc + static_cast<uint64_t>(((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4);
                                umma_bf16(tmem + 256 * half, ad, bslot + static_cast<uint64_t>((k4 * 8192) >> 4), kIdPV,
                                          (first && kk == 0) ? 0u : 1u);
                            }
                            umma_commit(&misc->v_empty[s]);
                            MLA_TRACE_UNIT1(1, vcount);
                            ++vcount;
                        }
                        if (half == 0) MLA_TRACE_EVENT(2, tcount);
                    }
                    if (!ok) break;
                    if (partial) ++zcount;   // partial tiles seen
                    umma_commit(&misc->pv_done[buf]);
                    MLA_TRACE_EVENT(6, tcount);
                    ++tcount;
                    PAIR_PROGRESS(4, tcount);
                    more = cur.advance(new_seg);
                }
            }
        } else if (warp >= 4) {
            // ---------------------------------------------------------- correction / epilogue warpgroup
            const int h = threadIdx.x - 128;
            const uint32_t lane_base = static_cast<uint32_t>(warp - 4) * 32;
            const uint32_t s_pempty = mapa_shared(smem_u32(&misc->p_empty[0]), partner);
            // requests with no tokens: out = 0, lse = -inf
            for (int si = seg_begin; si < seg_end; ++si) {
                const Segment sg = prm.segments[si];
                if (sg.t_end > sg.t_begin) continue;
                const size_t o0 = static_cast<size_t>(sg.b) * hq * kDimCkv;
                for (int i = h; i < hq * kDimCkv / 4; i += 128)
                    st_out4(final_out(prm), o0 + 4 * static_cast<size_t>(i), make_float4(0.f, 0.f, 0.f, 0.f));
                if (h < hq) prm.lse[static_cast<size_t>(sg.b) * hq + h] = -INFINITY;
            }
            uint32_t tcount = 0, vcount = 0, zcount = 0;
            bool ok = true;
            for (int si = seg_begin; si < seg_end && ok; ++si) {
                const Segment sg = prm.segments[si];
                if (sg.t_end <= sg.t_begin) continue;
                for (int t0 = sg.t_begin; t0 < sg.t_end && ok; t0 += C::kTile) {
                    const int ntok = min(C::kTile, sg.t_end - t0);
                    const bool first = t0 == sg.t_begin, last = t0 + C::kTile >= sg.t_end;
                    const int nv = (ntok + 63) / 64;
                    const uint32_t buf = tcount % C::kPBufs, ub = tcount / C::kPBufs;
                    ok = pair_wait<true>(&misc->p_full[buf], ub & 1, misc, partner_abort, prm.status, 61);
                    ok = !named_barrier_or(1, 128, !ok || aborted());
                    if (!ok) break;
                    if (h == 0) MLA_TRACE_EVENT(3, tcount);
                    // everything rank 0 left with this P buffer is read before the buffer goes back
                    const PairHand* hd = pair_hand(smem + C::kOffP + buf * C::kPBufBytes);
                    const bool resc = !first && *reinterpret_cast<const volatile int*>(&hd->rescale[0]);
                    const float alpha = hd->alpha[h];
                    const float fin_m = last ? hd->fin_m[h] : 0.f;
                    const float fin_l = last ? hd->fin_l[h] : 1.f;
                    // value rows [ntok, next multiple of 16) of the partial 64-token slot of one half:
                    // stale or NaN page tails the step's MMA would otherwise read.  The MMA thread
                    // raises vz_go[half] once that slot has landed (it is the ring's consumer; these
                    // warps could not tell the slot's phase apart from its previous use's).
                    auto zero_half = [&](int half) {
                        const int qz = ntok >> 6, r_lo = ntok & 63, r_hi = (r_lo + 15) & ~15;
                        const uint32_t vi = vcount + half * nv + qz;
                        ok = pair_wait(&misc->vz_go[half], zcount & 1, misc, partner_abort, prm.status, 62);
                        if (ok) {
                            uint8_t* slot = smem + C::kOffV + (vi % C::kVSlots) * C::kVSlotBytes;
                            for (int i = h; i < (r_hi - r_lo) * 32; i += 128) {
                                const int r = r_lo + i / 32, c = (i / 8) & 3, u = i & 7;
                                *reinterpret_cast<uint4*>(slot + (r >> 3) * 4096 + c * 1024 + (r & 7) * 128 + u * 16) =
                                    make_uint4(0, 0, 0, 0);
                            }
                        }
                        fence_proxy_async_smem();
                        ok = !named_barrier_or(1, 128, !ok || aborted());
                        if (ok && h == 0) mbar_arrive(&misc->vz_done[half]);
                    };
                    if (resc) {
                        // O row *= alpha once the previous tile's O += P V has completed.  The TMEM
                        // accesses are warp-collective: a warp takes the branch when any of its
                        // heads moved, each lane scaling by its own factor (1 if unchanged).
                        if (__any_sync(0xffffffffu, alpha != 1.f)) {
                            tc_fence_after();
#pragma unroll 1
                            for (int c = 0; c < 512; c += 32) {
                                uint32_t r[32];
                                tmem_ld32(tmem_addr(tmem, lane_base, c), r);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                                tmem_st32(tmem_addr(tmem, lane_base, c), r);
                            }
                            tmem_wait_st();
                        }
                        tc_fence_before();
                        named_barrier_sync(1, 128);
                        if (h == 0) mbar_arrive(&misc->corr_done);
                    }
                    if (ntok & 15) {   // after the rescale: the MMA thread signals only once past corr_done
                        zero_half(0);
                        if (ok) zero_half(1);
                        if (!ok) break;
                        ++zcount;
                    }
                    vcount += 2 * nv;
                    // this tile's O += P V done: its P buffer goes back to rank 0
                    ok = pair_wait(&misc->pv_done[buf], ub & 1, misc, partner_abort, prm.status, 63);
                    ok = !named_barrier_or(1, 128, !ok || aborted());
                    if (!ok) break;
                    if (h == 0) mbar_arrive_cluster(s_pempty + buf * 8);
                    if (h == 0) MLA_TRACE_EVENT(7, tcount);
                    ++tcount;
                    if (h == 0) PAIR_PROGRESS(5, tcount);
                    if (!last) continue;
                    // ---- epilogue: O / l -> out (or the piece's partial), lse
                    tc_fence_after();
                    const float inv = 1.f / fin_l;
                    const float lse_h = (fin_m + log2f(fin_l)) * 0.69314718055994530942f;
                    OutDst od;
                    size_t orow;
                    float* lbase;
                    if (sg.slot < 0) {
                        od = final_out(prm);
                        orow = (static_cast<size_t>(sg.b) * hq + h) * kDimCkv;
                        lbase = prm.lse + static_cast<size_t>(sg.b) * hq;
                    } else {
                        od = fp32_dst(prm.part_o);
                        orow = (static_cast<size_t>(sg.slot) * hq + h) * kDimCkv;
                        lbase = prm.part_lse + static_cast<size_t>(sg.slot) * hq;
                    }
#pragma unroll 1
                    for (int c = 0; c < 512; c += 32) {   // the TMEM loads are warp-collective: every lane
                        uint32_t r[32];
                        tmem_ld32(tmem_addr(tmem, lane_base, c), r);
                        tmem_wait_ld();
                        if (h < hq) {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                st_out4(od, orow + c + 4 * i,
                                        make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                                    __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv));
                        }
                    }
                    if (h < hq) lbase[h] = lse_h;
                    tc_fence_before();
                    named_barrier_sync(1, 128);
                    if (h == 0) mbar_arrive(&misc->epi_done);
                    if (sg.slot >= 0) {
                        // split request: the last piece to arrive merges all of them in slot order
                        __threadfence();
                        named_barrier_sync(1, 128);
                        if (h == 0) misc->merge_flag = (atomicAdd(&prm.counters[sg.item], 1) == sg.n_slots - 1);
                        named_barrier_sync(1, 128);
                        if (misc->merge_flag) {
                            __threadfence();
                            merge_split_pieces<HQ, 128>(prm, sg.b, sg.slot_begin, sg.n_slots, 0, h, 1, misc->mrg_max,
                                                        misc->mrg_inv, misc->mrg_w);
                            if (h == 0) prm.counters[sg.item] = 0;
                        }
                        named_barrier_sync(1, 128);
                    }
                }
            }
        }
    }

    if (threadIdx.x == 0) PAIR_PROGRESS(6, 1000000 + misc->abort_flag);
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    cluster_sync();   // no CTA leaves while its partner may still write into its shared memory
    if (threadIdx.x == 0) PAIR_PROGRESS(7, 1);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace mla
