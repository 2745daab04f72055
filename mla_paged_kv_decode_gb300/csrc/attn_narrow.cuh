// MLA paged decode attention over a bf16 latent cache for narrow head counts (16 or 32
// query heads per CTA) on sm_103a: TMA page staging into an mbarrier ring, tensor-core math
// with warp-level mma.sync (m16n8k16, bf16 in, fp32 accumulate).
//
// Why warp MMA here: the score contraction of a 16-head request has 16 rows per query, and a
// tcgen05.mma of M 128 has a floor (one of N 64 costs about what one of N 128 does, ~64 SM
// cycles, measured on this GPU), so tcgen05 tiles of 128 tokens x 16 heads would take 68
// instructions per tile (~34 cycles per token at that floor) with TMEM round trips for the
// softmax in between.  The warp MMA has no such floor: 16 heads x 1088 MACs per cached token
// is ~17 cycles per token per SM, against the ~49 cycles per token an SM may spend at full
// HBM bandwidth.  The 64/128-head path (attn_pair.cuh) and the e4m3 cache (attn_e4m3.cuh) run
// on tcgen05.
//
// Absorbed MLA decode is MQA with one KV head: key [ckv | kpe] (576), value ckv (512)
// ("Benchmarking MLA", FlashInfer issue #700).  The layout of the work follows the split-K
// idea of FlashMLA PR #233's sm86 kernel ("Q in registers, split-K QK inside the CTA, a
// multi-stage ... KV ring"), rebuilt for TMA and the GB300 memory system:
//
//   * a CTA owns HG heads of every segment of its plan slot and walks it in 32-token tiles,
//     one ring stage each (36 KB: 8 ckv chunks of 64 dims + kpe, 128-byte swizzle; one 3-D
//     TMA box per stage when a page holds it, else one 2-D box per chunk and page piece);
//   * warpgroup 0 is the producer (warp 0 issues the copies); two compute groups of 4 warps
//     take the math.  With 16 heads the groups take alternate tiles of a segment (token
//     groups) and merge their (m, l, O) at its end; with 32 heads each group takes 16 heads;
//   * in a group, warp k holds q for dims [144k, 144k + 144) in registers and computes the
//     partial scores of the tile over those dims; the 4 partials go through shared memory
//     and warp k finishes the scores of tokens [8k, 8k + 8);
//   * the online softmax keeps a lazy running max (moved, and O rescaled, only when a tile
//     exceeds it by more than 2^8), P goes through shared memory as bf16 A fragments, and
//     warp k accumulates O += P V for its own 128 latent dims (V read with ldmatrix.trans).
//
// A split request's pieces write normalised partials; the last CTA to finish one merges them
// in slot order (FlashMLA PR #233, "deterministic combine"; attn.cuh).  Every mbarrier wait
// is bounded.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace mla {

constexpr int kNarrowTile = 32;        // tokens per tile (= one ring stage)
constexpr int kNarrowStageTok = 32;    // tokens per ring stage

template <int HG>
struct NarrowCfg {
    static_assert(HG == 16 || HG == 32, "heads per CTA");
    static constexpr int kHeadGroups = HG / 16;               // 16-head groups
    static constexpr int kTokenGroups = (HG == 16) ? 2 : 1;   // groups taking alternate tiles
    static constexpr int kGroups = kHeadGroups * kTokenGroups; // 4-warp compute groups
    static constexpr int kComputeWarps = 4 * kGroups;          // 8 in both cases: 2 warps per SM sub-partition
    // warpgroup 0: the TMA producer (warp 0; warps 1-3 idle); warpgroups 1 and 2: the compute
    // groups.  Launched at 168 registers a thread (65536 / 384); warpgroup 0 gives registers
    // back and the compute warpgroups take them (128 x 80 + 256 x 208 <= 384 x 168).
    static constexpr int kProducerWarps = 4;
    // Warps 0 and 1 issue the copies: one issuing thread starts about one ring stage per ~0.45 us
    // (measured on this GPU), so two of them keep more of the ring in flight.  Producer p owns
    // the stages s with s % kIssuers == p, so every stage has one issuer.
    static constexpr int kIssuers = 2;
    static constexpr int kThreads = 32 * (kProducerWarps + kComputeWarps);
    static constexpr uint32_t kProducerRegs = 80;
    static constexpr uint32_t kComputeRegs = 208;
    static_assert(128 * kProducerRegs + 32 * kComputeWarps * kComputeRegs <= 65536 / kThreads / 8 * 8 * kThreads,
                  "register split");
    // ring stages, filled by TMA: 8 value chunks (64 dims x 32 tokens, 128-byte swizzle) + the
    // kpe chunk = 36 KB
    static constexpr int kChunkBytes = kNarrowStageTok * 128;  // 4 KB: 32 rows of 128 B
    static constexpr int kKpeOff = 8 * kChunkBytes;
    static constexpr int kStageBytes = 9 * kChunkBytes;
    static constexpr int kStages = 5;
    static constexpr int kStageLoadBytes = kNarrowStageTok * 1152;
    static constexpr int kPartBytes = 4 * 32 * 16 * 4;         // per group: 4 warps x 32 lanes x 16 floats = 8 KB
    static constexpr int kPRowBytes = 80;                       // P row: 32 16-bit tokens + 16 B pad (conflict-free ldmatrix)
    static constexpr int kGroupScratch = 16 * kPRowBytes + 4 * 16 * 4;   // P tile + per-warp row maxima
    static constexpr int kOffStage = 0;
    static constexpr int kOffPart = kOffStage + kStages * kStageBytes;
    static constexpr int kOffScratch = kOffPart + kGroups * kPartBytes;
    static constexpr int kOffMisc = kOffScratch + kGroups * kGroupScratch;
    static constexpr int kMiscBytes = 3072;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;
    static_assert(kStageBytes % 1024 == 0, "stage layout");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    // the token-group merge passes one group's O (16 heads x 512 dims fp32) in two halves
    // through the partial-score buffers of both groups
    static_assert(kTokenGroups == 1 || 2 * kGroups * kPartBytes >= 16 * kDimCkv * 4, "merge buffer");
};

struct NarrowMisc {
    uint64_t full[5], empty[5];
    int abort_flag;
    int merge_flag[2];
    float mrg_max[2][16];
    float mrg_inv[2][16];
    float mrg_w[2][128];
    float tg_m[16], tg_l[16];   // token-group merge: running max and row sum of group 1
};

// Debug builds (MLA_TRACE): a timestamp at step k of a segment switch of the traced CTA, per
// token group, in the per-unit area of the trace buffer.
#ifdef MLA_TRACE
#define NARROW_STAMP(k)                                                                                   \
    do {                                                                                                  \
        if (prm.trace && blockIdx.x == MLA_TRACE_FIRST && kr == 0 && lane == 0 && si - seg_begin < 16)     \
            prm.trace[2 * 8 * 256 + (tg * 16 + (k)) * 16 + (si - seg_begin)] = global_timer_ns();         \
    } while (0)
#else
#define NARROW_STAMP(k) \
    do {                \
    } while (0)
#endif

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}


__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void mma_f16_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// The 16-bit input format of the narrow kernel: bf16, or (F16) IEEE fp16 q, ckv and kpe.  P
// takes the same format (the MMA's operands share one type); it lies in [0, 2^8].
template <bool F16>
__device__ __forceinline__ void mma16_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    if constexpr (F16)
        mma_f16_16816(c, a, b0, b1);
    else
        mma_bf16_16816(c, a, b0, b1);
}

template <bool F16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
    if constexpr (F16)
        return pack_f16(lo, hi);
    else
        return pack_bf16(lo, hi);
}

// Address of the 16-byte unit holding (row, dims 8u..8u+7) of a 64-dim chunk stored as
// rows of 128 bytes with the 128-byte swizzle (unit index XOR row % 8).
__device__ __forceinline__ uint32_t sw_unit(uint32_t chunk_base, uint32_t row, uint32_t unit) {
    return chunk_base + row * 128 + ((unit ^ (row & 7)) << 4);
}

template <int HG, bool F16 = false>
__global__ void __launch_bounds__(NarrowCfg<HG>::kThreads, 1)
    mla_decode_narrow_kernel(const __grid_constant__ CUtensorMap tm_ckv, const __grid_constant__ CUtensorMap tm_kpe,
                             const AttnParams prm, const uint16_t* __restrict__ q_nope,
                             const uint16_t* __restrict__ q_pe) {
    using C = NarrowCfg<HG>;
    static_assert(sizeof(NarrowMisc) <= C::kMiscBytes && C::kStages <= 5, "misc region");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stage_base = smem + C::kOffStage;
    float* part_base = reinterpret_cast<float*>(smem + C::kOffPart);
    NarrowMisc* misc = reinterpret_cast<NarrowMisc*>(smem + C::kOffMisc);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int unit = blockIdx.x / prm.head_groups;
    const int group_cta = blockIdx.x % prm.head_groups;
    const int seg_begin = prm.unit_ptr[unit];
    const int seg_end = prm.unit_ptr[unit + 1];
    const int P = prm.page_size;
    const int box_rows = P < kNarrowStageTok ? P : kNarrowStageTok;

    // Prologue before the previous kernel in the stream has finished (programmatic dependent
    // launch): barrier set-up and this CTA's slice of the plan, which only the plan commit
    // writes.  Every read of the caller's buffers and every write comes after grid_dep_wait.
    grid_dep_launch();
    if (threadIdx.x == 0) {
        MLA_TRACE_CTA(0);
#ifdef MLA_TRACE
        if (prm.trace) {
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            prm.trace[4 * 8 * 256 + blockIdx.x * 8 + 7] = smid;
        }
#endif
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&misc->full[i], 1);
            // released by the 4 warps of every 16-head group that consumes the stage: one token
            // group takes each tile, and all kHeadGroups head groups read it
            mbar_init(&misc->empty[i], 4 * C::kHeadGroups);
        }
        misc->abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_ckv);
        prefetch_tensormap(&tm_kpe);
    }
    __syncthreads();
    grid_dep_wait();

    if (warp < C::kProducerWarps) regs_dec<C::kProducerRegs>();
    else regs_inc<C::kComputeRegs>();

    if (warp < C::kIssuers) {
        // ------------------------------------------------------------ TMA producers
        const int pid = warp;
        uint32_t scount = 0, tile_idx = 0;
        bool ok = true;
        TileCursorT<kNarrowTile> cur;
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
            const int nst = (ntok + kNarrowStageTok - 1) / kNarrowStageTok;
            for (int st = 0; st < nst && ok; ++st) {
                const int t_st = cur.t0 + st * kNarrowStageTok;                   // first token of the stage
                const int n_st = min(kNarrowStageTok, cur.sg.t_end - t_st);        // tokens in the stage
                const int nbox = (n_st + box_rows - 1) / box_rows;
                const int first_page = t_st / P;
                const int last_page_st = (t_st + nbox * box_rows - 1) / P;
                if (last_page_st + 1 > win_base + 32 || first_page < win_base) {
                    const int seg_last_page = (cur.sg.t_end - 1) / P;
                    win_base = first_page;
                    win_page = (win_base + lane <= seg_last_page) ? pages[win_base + lane] : 0;
                }
                const uint32_t s = scount % C::kStages, use = scount / C::kStages;
                if (static_cast<int>(s) % C::kIssuers != pid) {   // the other producer's stage
                    ++scount;
                    continue;
                }
                uint64_t* bar_full = &misc->full[s];
                if (lane == 0 && use > 0) ok = wait_phase_flag(&misc->empty[s], (use - 1) & 1, &misc->abort_flag, prm.status, 21);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
#ifdef MLA_TEST_HOOKS
                // test builds: CTA 0 never fills its first stage, so the bounded wait on it runs out
                if (prm.test_withhold && blockIdx.x == 0 && scount == 0) {
                    ++scount;
                    continue;
                }
#endif
                uint8_t* dst = stage_base + s * C::kStageBytes;
                // bytes per token: bf16 ckv + kpe = 1152
                if (lane == 0)
                    mbar_arrive_expect_tx(bar_full, static_cast<uint32_t>(nbox * box_rows * (C::kStageLoadBytes / kNarrowStageTok)));
                if (lane == 0) MLA_TRACE_EVENT(pid, tile_idx);
                for (int bx = 0; bx < nbox; ++bx) {
                    const int t = t_st + bx * box_rows;
                    const int pg = __shfl_sync(0xffffffffu, win_page, (t / P - win_base) & 31);
                    if (lane == 0) {
                        const int y = pg * P + (t % P);
                        if (box_rows == kNarrowStageTok) {
                            // all 8 ckv chunks in one 3-D box (64 dims, 32 rows, 8 chunks), which lands as
                            // [chunk][row][128 B] -- the stage layout the ldmatrix addressing expects
                            tma_load_3d(dst, &tm_ckv, &misc->full[s], 0, y, 0);
                        } else {
                            for (int c = 0; c < 8; ++c)
                                tma_load_2d(dst + c * C::kChunkBytes + bx * box_rows * 128, &tm_ckv, &misc->full[s],
                                            c * 64, y);
                        }
                        tma_load_2d(dst + 8 * C::kChunkBytes + bx * box_rows * 128, &tm_kpe, &misc->full[s], 0, y);
                    }
                }
                ++scount;
            }
            ++tile_idx;
            more = cur.advance(new_seg);
        }
        if (lane == 0) {   // this producer's stages: every copy lands before the CTA can exit
            if (pid == 0) MLA_TRACE_CTA(1);
            const uint64_t t0 = global_timer_ns();
            for (int s = pid; s < C::kStages; s += C::kIssuers) {
                const uint32_t uses = scount / C::kStages + (static_cast<uint32_t>(s) < scount % C::kStages ? 1 : 0);
                if (uses == 0) continue;
                while (!mbar_try_wait(&misc->full[s], (uses - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
            }
        }
    } else if (warp >= C::kProducerWarps) {
        // ------------------------------------------------------------ compute warps
        const int cw = warp - C::kProducerWarps;  // 0 .. kComputeWarps-1
        const int grp = cw / 4;                  // compute group (4 warps)
        const int hgi = grp / C::kTokenGroups;   // 16-head group within the CTA
        const int tg = grp % C::kTokenGroups;    // token group: takes tiles t with t % kTokenGroups == tg
        const int kr = cw % 4;                   // score split: dims [144 kr, 144 kr + 144); PV: dims [128 kr, +128)
        const int g = lane >> 2, c4 = lane & 3;  // mma fragment row group / column pair
        const uint32_t named_bar = 1 + grp;      // 4-warp group barrier
        const uint32_t merge_bar = 1 + C::kGroups + hgi;   // both token groups of a head group
        const int head0 = group_cta * HG + hgi * 16;   // first head of this warp's group
        const uint32_t stage0 = smem_u32(stage_base);
        float* part = part_base + grp * (C::kPartBytes / 4);
        uint8_t* pbuf = smem + C::kOffScratch + grp * C::kGroupScratch;              // P tile [16][80 B]
        float* rowmax = reinterpret_cast<float*>(pbuf + 16 * C::kPRowBytes);           // [4 warps][16 rows]
        uint32_t scount = 0;     // ring stages consumed so far by the CTA (both token groups)
        bool ok = true;
        // q fragments for dims [144 kr, 144 kr + 144): 9 k-steps of 16 (dims >= 512 are q_pe)
        uint32_t qa[9][4];
        auto load_q = [&](int b) {
            const size_t qrow0 = static_cast<size_t>(b) * prm.h_q + head0;
#pragma unroll
            for (int ks = 0; ks < 9; ++ks) {
                const int kd = kr * 144 + ks * 16;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int row = g + ((r & 1) ? 8 : 0);
                    const int dim = kd + 2 * c4 + ((r & 2) ? 8 : 0);   // fragment k index 2 c4 + {0, 1} (+ 8)
                    const uint16_t* src = dim < kDimCkv ? q_nope + (qrow0 + row) * kDimCkv + dim
                                                        : q_pe + (qrow0 + row) * kDimKpe + (dim - kDimCkv);
                    qa[ks][r] = *reinterpret_cast<const uint32_t*>(src);
                }
            }
        };
        for (int si = seg_begin; si < seg_end && ok; ++si) {
            const Segment sg = prm.segments[si];
            if (sg.t_end <= sg.t_begin) {
                if (tg == 0) {
                    const size_t o0 = (static_cast<size_t>(sg.b) * prm.h_q + head0) * kDimCkv;
                    for (int i = kr * 32 + lane; i < 16 * kDimCkv; i += 128) st_out(final_out(prm), o0 + i, 0.f);
                    if (kr == 0 && lane < 16) prm.lse[static_cast<size_t>(sg.b) * prm.h_q + head0 + lane] = -INFINITY;
                }
                continue;
            }
            load_q(sg.b);
#ifdef MLA_TRACE
            if (prm.trace && blockIdx.x == MLA_TRACE_FIRST && kr == 0 && lane == 0 && si - seg_begin < 16) {
                uint64_t t_;   // stamped once this thread's query words have arrived
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_) : "r"(qa[8][3]), "r"(qa[0][0]));
                prm.trace[2 * 8 * 256 + (tg * 16 + 1) * 16 + (si - seg_begin)] = t_;
            }
#endif

            float o[16][4];
#pragma unroll
            for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            float m_run[2] = {-INFINITY, -INFINITY};   // rows g and g + 8 (log2 domain)
            float l_part[2] = {0.f, 0.f};
            int tile_in_seg = 0;
            for (int t0 = sg.t_begin; t0 < sg.t_end; t0 += kNarrowTile, ++tile_in_seg) {
                const int ntok = min(kNarrowTile, sg.t_end - t0);
                if (tile_in_seg % C::kTokenGroups != tg) {   // the other token group's tile
                    ++scount;
                    continue;
                }
                const uint32_t sl = scount % C::kStages;
                const uint32_t use = scount / C::kStages;
                // With two token groups the stages are consumed by the groups in turn: this
                // stage's previous use (5 tiles back) is the other group's tile, which may not
                // have landed yet, and a parity wait on the full barrier alone could then match
                // that older phase.  So wait first until the previous use is released (its
                // empty-barrier phase): the use before it (10 tiles back) is this group's own
                // tile or from a segment both groups have finished, so that empty barrier is in
                // the previous use's phase or this one and the wait is unambiguous.  Once the
                // previous use is released the full barrier is in this use's phase.
                // One warp of the group waits; the group barrier after it orders the other warps'
                // reads of the stage after that warp's observation of the completed copy.
                if (kr == 0) {
                    if (C::kTokenGroups > 1 && use > 0)
                        ok = wait_phase_flag(&misc->empty[sl], (use - 1) & 1, &misc->abort_flag, prm.status, 23);
                    if (ok) ok = wait_phase_flag(&misc->full[sl], use & 1, &misc->abort_flag, prm.status, 22);
                }
                const uint32_t st_addr = stage0 + sl * C::kStageBytes;
                ok = !named_barrier_or(named_bar, 128, !ok || *reinterpret_cast<volatile int*>(&misc->abort_flag));
                if (!ok) break;
                if (kr == 0 && lane == 0) MLA_TRACE_EVENT(tg ? 6 : 2, scount);
                // ---- partial scores over this warp's 144 dims for the 4 n8 token tiles
                float sc[4][4];
#pragma unroll
                for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 9; ++ks) {
                    const int kd = kr * 144 + ks * 16;
                    // 16-dim step: latent or rope
                    const uint32_t chunk_base = kd < kDimCkv ? st_addr + (kd >> 6) * C::kChunkBytes
                                                             : st_addr + C::kKpeOff;
                    const int unit0 = (kd & 63) >> 3;          // 16-byte unit of the k-step's first 8 dims
                    uint32_t bf[2][4];
#pragma unroll
                    for (int np = 0; np < 2; ++np) {           // pairs of n8 tiles = 16 tokens
                        const int tok = np * 16 + (lane & 7) + ((lane & 16) ? 8 : 0);
                        ldsm_x4(sw_unit(chunk_base, tok, unit0 + ((lane & 8) ? 1 : 0)),
                                bf[np][0], bf[np][1], bf[np][2], bf[np][3]);
                    }
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        if (np * 16 < ntok) {
                            mma16_16816<F16>(sc[2 * np], qa[ks], bf[np][0], bf[np][1]);
                            mma16_16816<F16>(sc[2 * np + 1], qa[ks], bf[np][2], bf[np][3]);
                        }
                    }
                }
                // ---- exchange partials within the group; warp kr finishes the scores of n8 tile kr
                {
                    float4* dst = reinterpret_cast<float4*>(part) + kr * 4 * 32;
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i * 32 + lane] = make_float4(sc[i][0], sc[i][1], sc[i][2], sc[i][3]);
                }
                // zero the value rows of a partial 16-token step (stale or NaN bytes past the last
                // token): 8 chunks of 128 B per row
                if (ntok < kNarrowTile && (ntok & 15)) {
                    const int r_end = (ntok + 15) & ~15;
                    for (int tok = ntok + kr; tok < r_end; tok += 4) {
                        uint4* rowp = reinterpret_cast<uint4*>(stage_base + (st_addr - stage0) + tok * 128);
                        for (int c = 0; c < 8; ++c) rowp[c * (C::kChunkBytes / 16) + (lane & 7)] = make_uint4(0, 0, 0, 0);
                    }
                }
                named_barrier_sync(named_bar, 128);
                if (cw == 0 && lane == 0) MLA_TRACE_EVENT(3, scount);
                float s4[4];   // scores of (row g, tokens 8kr + 2c4, +1) and (row g + 8, same tokens)
                {
                    const float4* src = reinterpret_cast<const float4*>(part);
                    const float4 a0 = src[(0 * 4 + kr) * 32 + lane], a1 = src[(1 * 4 + kr) * 32 + lane];
                    const float4 a2 = src[(2 * 4 + kr) * 32 + lane], a3 = src[(3 * 4 + kr) * 32 + lane];
                    s4[0] = ((a0.x + a1.x) + a2.x) + a3.x;
                    s4[1] = ((a0.y + a1.y) + a2.y) + a3.y;
                    s4[2] = ((a0.z + a1.z) + a2.z) + a3.z;
                    s4[3] = ((a0.w + a1.w) + a2.w) + a3.w;
                }
                if (ntok < kNarrowTile) {
                    const int tok = kr * 8 + 2 * c4;
                    if (tok >= ntok) s4[0] = s4[2] = -INFINITY;
                    if (tok + 1 >= ntok) s4[1] = s4[3] = -INFINITY;
                }
                // ---- row maxima of the tile (raw scores; sm_scale > 0 keeps the order)
                float mt[2] = {fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3])};
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mt[r] = fmaxf(mt[r], __shfl_xor_sync(0xffffffffu, mt[r], 1));
                    mt[r] = fmaxf(mt[r], __shfl_xor_sync(0xffffffffu, mt[r], 2));
                }
                if (c4 == 0) {
                    rowmax[kr * 16 + g] = mt[0];
                    rowmax[kr * 16 + g + 8] = mt[1];
                }
                named_barrier_sync(named_bar, 128);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int row = g + 8 * r;
                    const float m4 = fmaxf(fmaxf(rowmax[row], rowmax[16 + row]), fmaxf(rowmax[32 + row], rowmax[48 + row]));
                    // lazy running max (log2 units): move it, and rescale O and l, only when the tile max
                    // exceeds it by more than 8; every warp of the group takes the same decision
                    const float ms = m4 * prm.scale_log2;
                    if (ms > m_run[r] + 8.f) {
                        const float alpha = fast_exp2(m_run[r] - ms);
                        m_run[r] = ms;
                        l_part[r] *= alpha;
#pragma unroll
                        for (int n = 0; n < 16; ++n) {
                            o[n][2 * r] *= alpha;
                            o[n][2 * r + 1] *= alpha;
                        }
                    }
                }
                {
                    const float p0 = fast_exp2(fmaf(s4[0], prm.scale_log2, -m_run[0]));
                    const float p1 = fast_exp2(fmaf(s4[1], prm.scale_log2, -m_run[0]));
                    const float p2 = fast_exp2(fmaf(s4[2], prm.scale_log2, -m_run[1]));
                    const float p3 = fast_exp2(fmaf(s4[3], prm.scale_log2, -m_run[1]));
                    l_part[0] += p0 + p1;
                    l_part[1] += p2 + p3;
                    const uint32_t w0 = pack16<F16>(p0, p1), w1 = pack16<F16>(p2, p3);
                    *reinterpret_cast<uint32_t*>(pbuf + g * C::kPRowBytes + (kr * 8 + 2 * c4) * 2) = w0;
                    *reinterpret_cast<uint32_t*>(pbuf + (g + 8) * C::kPRowBytes + (kr * 8 + 2 * c4) * 2) = w1;
                }
                named_barrier_sync(named_bar, 128);
                uint32_t pa[2][4];   // P as the A operand of the 2 k16 token steps
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const int prow = (lane & 7) + ((lane & 8) ? 8 : 0);
                    const int pcol = kt * 16 + ((lane & 16) ? 8 : 0);
                    ldsm_x4(smem_u32(pbuf) + prow * C::kPRowBytes + pcol * 2, pa[kt][0], pa[kt][1], pa[kt][2], pa[kt][3]);
                }
                if (cw == 0 && lane == 0) MLA_TRACE_EVENT(4, scount);
                // ---- O[16 x 128 dims of this warp] += P V
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    if (kt * 16 >= ntok) break;
                    const int tok = kt * 16 + (lane & 7) + ((lane & 8) ? 8 : 0);
                    uint32_t vf[8][4];
#pragma unroll
                    for (int dp = 0; dp < 8; ++dp) {          // pairs of n8 dim tiles = 16 dims
                        const int d0 = kr * 128 + dp * 16;
                        const int unit = ((d0 & 63) >> 3) + ((lane & 16) ? 1 : 0);
                        ldsm_x4_t(sw_unit(st_addr + (d0 >> 6) * C::kChunkBytes, tok, unit), vf[dp][0], vf[dp][1],
                                  vf[dp][2], vf[dp][3]);
                    }
#pragma unroll
                    for (int dp = 0; dp < 8; ++dp) {
                        mma16_16816<F16>(o[2 * dp], pa[kt], vf[dp][0], vf[dp][1]);
                        mma16_16816<F16>(o[2 * dp + 1], pa[kt], vf[dp][2], vf[dp][3]);
                    }
                }
                __syncwarp();
                if (kr == 0 && lane == 0) MLA_TRACE_EVENT(tg ? 7 : 5, scount);
                if (lane == 0) mbar_arrive(&misc->empty[sl]);
                ++scount;
            }

            if (C::kTokenGroups == 2) {
                // Both token groups meet at every segment end, also after a bounded wait ran out,
                // and leave together: neither can then block in the cross-group barriers below
                // waiting for a group that has left.
                ok = !named_barrier_or(merge_bar, 256, !ok || *reinterpret_cast<volatile int*>(&misc->abort_flag));
            }
            if (!ok) break;
            NARROW_STAMP(6);   // both token groups at the segment end
            if (kr == 0 && lane == 0) MLA_TRACE_CTA(2 + grp);
            // A split piece takes its arrival ticket now; the atomic's round trip overlaps the
            // row sums and the token-group merge below, and only the ticket's use waits for it.
            const int gt = kr * 32 + lane;   // 0..127 within the group
            const int ctr = (sg.item * prm.head_groups + group_cta) * C::kHeadGroups + hgi;
            int ticket = 0;
            if (sg.slot >= 0 && tg == 0 && gt == 0) ticket = atomicAdd(&prm.counters[ctr], 1);
            // ---- row sums: quad, then the 4 warps of the group (each summed its own 8 tokens per tile)
            float l[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                l[r] = l_part[r];
                l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
                l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
            }
            named_barrier_sync(named_bar, 128);
            if (c4 == 0) {
                rowmax[kr * 16 + g] = l[0];
                rowmax[kr * 16 + g + 8] = l[1];
            }
            named_barrier_sync(named_bar, 128);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int row = g + 8 * r;
                l[r] = (rowmax[row] + rowmax[16 + row]) + (rowmax[32 + row] + rowmax[48 + row]);
            }
            NARROW_STAMP(5);   // row sums
            if (C::kTokenGroups == 2) {
                // ---- merge the two token groups: group 1 passes (O, m, l) to group 0 through shared
                // memory (the partial-score buffers of both groups, two halves of O), group 0 combines
                float4* xo = reinterpret_cast<float4*>(part_base + (hgi * C::kTokenGroups) * (C::kPartBytes / 4));
                named_barrier_sync(merge_bar, 256);
                if (tg == 1 && kr == 0 && c4 == 0) {
                    misc->tg_m[g] = m_run[0];
                    misc->tg_m[g + 8] = m_run[1];
                    misc->tg_l[g] = l[0];
                    misc->tg_l[g + 8] = l[1];
                }
                float w0[2] = {1.f, 1.f}, w1[2] = {0.f, 0.f};
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (tg == 1) {
#pragma unroll
                        for (int n = 0; n < 8; ++n)
                            xo[(kr * 8 + n) * 32 + lane] =
                                make_float4(o[half * 8 + n][0], o[half * 8 + n][1], o[half * 8 + n][2], o[half * 8 + n][3]);
                    }
                    named_barrier_sync(merge_bar, 256);
                    if (tg == 0) {
                        if (half == 0) {
                            const float m1[2] = {misc->tg_m[g], misc->tg_m[g + 8]};
                            const float l1[2] = {misc->tg_l[g], misc->tg_l[g + 8]};
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const float mm = fmaxf(m_run[r], m1[r]);
                                w0[r] = exp2f(m_run[r] - mm);
                                w1[r] = (m1[r] == -INFINITY) ? 0.f : exp2f(m1[r] - mm);
                                m_run[r] = mm;
                                l[r] = l[r] * w0[r] + l1[r] * w1[r];
                            }
                        }
#pragma unroll
                        for (int n = 0; n < 8; ++n) {
                            const float4 v = xo[(kr * 8 + n) * 32 + lane];
                            float* on = o[half * 8 + n];
                            on[0] = on[0] * w0[0] + v.x * w1[0];
                            on[1] = on[1] * w0[0] + v.y * w1[0];
                            on[2] = on[2] * w0[1] + v.z * w1[1];
                            on[3] = on[3] * w0[1] + v.w * w1[1];
                        }
                    }
                    named_barrier_sync(merge_bar, 256);   // the buffer is rewritten next
                }
            }
            NARROW_STAMP(0);   // token groups merged
            // At the unit's last segment token group 1 has no more tiles: if the segment is a
            // split piece it stays to merge with group 0 (256 threads, one round of loads)
            const bool wide = C::kTokenGroups == 2 && sg.slot >= 0 && si == seg_end - 1;
            if (tg == 1 && !wide) continue;
            if (tg == 0) {
                // ---- epilogue (token group 0): normalise and store this warp's 128 dims
                const float inv0 = 1.f / l[0], inv1 = 1.f / l[1];
                OutDst od;
                size_t o0;
                float* lbase;
                if (sg.slot < 0) {
                    od = final_out(prm);
                    o0 = (static_cast<size_t>(sg.b) * prm.h_q + head0) * kDimCkv;
                    lbase = prm.lse + static_cast<size_t>(sg.b) * prm.h_q + head0;
                } else {
                    od = fp32_dst(prm.part_o);
                    o0 = (static_cast<size_t>(sg.slot) * prm.h_q + head0) * kDimCkv;
                    lbase = prm.part_lse + static_cast<size_t>(sg.slot) * prm.h_q + head0;
                }
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    const int d = kr * 128 + n * 8 + 2 * c4;
                    st_out2(od, o0 + static_cast<size_t>(g) * kDimCkv + d, o[n][0] * inv0, o[n][1] * inv0);
                    st_out2(od, o0 + static_cast<size_t>(g + 8) * kDimCkv + d, o[n][2] * inv1, o[n][3] * inv1);
                }
                if (kr == 0 && c4 == 0) {
                    lbase[g] = (m_run[0] + log2f(l[0])) * 0.69314718055994530942f;
                    lbase[g + 8] = (m_run[1] + log2f(l[1])) * 0.69314718055994530942f;
                }
                NARROW_STAMP(2);   // epilogue stores issued
            }
            if (sg.slot >= 0) {
                // ---- split request: the piece with the last ticket merges all of them in slot order
                // (group 0 alone, or both token groups at the unit's last segment).  The others
                // publish their partial (stores, fence, then the ready count); the last one waits
                // until every other partial is published -- their CTAs hold tickets, so they are
                // running and wait on nothing -- and reads its own partial back after the group
                // barrier (same CTA), with no fence or second round trip on its path.
                const uint32_t mbar = wide ? merge_bar : named_bar;
                const uint32_t nthr = wide ? 256u : 128u;
                if (tg == 0 && gt == 0) misc->merge_flag[hgi] = (ticket == sg.n_slots - 1) ? 1 : 0;
                named_barrier_sync(mbar, nthr);
                NARROW_STAMP(3);   // ticket known
                if (!misc->merge_flag[hgi]) {
                    if (tg == 0) __threadfence();
                    NARROW_STAMP(7);   // partial stores fenced
                    named_barrier_sync(mbar, nthr);
                    if (tg == 0 && gt == 0) atomicAdd(&prm.ready[ctr], 1);
                } else {
                    if (tg == 0 && gt == 0) {
                        // an acquiring read of the count: the other pieces' partials are visible to this
                        // thread, and to the whole group after the barrier below
                        MLA_TRACE_CTA(4);
                        bool done = ld_acquire_gpu(prm.ready + ctr) >= sg.n_slots - 1;
                        const uint64_t t0 = global_timer_ns();
                        while (!done && !*reinterpret_cast<volatile int*>(&misc->abort_flag)) {
                            if (global_timer_ns() - t0 > kWaitLimitNs) {
                                misc->abort_flag = 1;
                                atomicCAS(prm.status, 0u, kStatusTimeout | 24u);
                                break;
                            }
                            done = ld_acquire_gpu(prm.ready + ctr) >= sg.n_slots - 1;
                        }
                        misc->merge_flag[hgi] = done ? 1 : 2;
                        MLA_TRACE_CTA(3);   // (debug builds) the other pieces are published
                    }
                    named_barrier_sync(mbar, nthr);
                    if (misc->merge_flag[hgi] == 1) {
                        if (wide)
                            merge_split_pieces_wide16(prm, sg.b, sg.slot_begin, sg.n_slots, head0, tg * 128 + gt,
                                                      merge_bar, named_bar, misc->mrg_max[hgi], misc->mrg_inv[hgi],
                                                      misc->mrg_w[hgi]);
                        else
                            merge_split_pieces<16, 128>(prm, sg.b, sg.slot_begin, sg.n_slots, head0, gt, named_bar,
                                                        misc->mrg_max[hgi], misc->mrg_inv[hgi], misc->mrg_w[hgi]);
                    }
                    if (tg == 0 && gt == 0) {
                        prm.counters[ctr] = 0;
                        prm.ready[ctr] = 0;
                        MLA_TRACE_CTA(5);
                    }
                }
                named_barrier_sync(mbar, nthr);
                NARROW_STAMP(4);   // published or merged
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) MLA_TRACE_CTA(6);
}

}  // namespace mla
