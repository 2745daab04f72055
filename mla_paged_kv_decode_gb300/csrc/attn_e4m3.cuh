// MLA paged decode attention over an 8-bit (e4m3) latent cache for 16 query heads per CTA
// on sm_103a: tcgen05 MMAs of kind::f8f6f4 with TMEM accumulators, tokens on the MMA's
// M axis.
//
// Absorbed MLA decode is MQA with one KV head: key [ckv | kpe] (576), value ckv (512)
// ("Benchmarking MLA", FlashInfer issue #700).  The cache keeps ckv as e4m3 codes with one
// fp32 scale per token and kpe in bf16, 644 bytes a token (FlashMLA PR #233, "FP8 e4m3 ...
// with one scale per token (644 instead of 1152 bytes per token), dequantized inside the
// kernel").  The codes are the tensor-core operands as they are:
//
//   S^T = K Q^T   M = 128 tokens, N = 32, K = 512: A = the tile's codes (K-major), B = the
//                 query as two e4m3 rows per head, q sigma = qh + ql exactly (sigma a power
//                 of two per head putting its largest |q| in [128, 256); every bf16 entry
//                 within 2^10 of that splits exactly: 4 significant bits in qh, the rest
//                 in ql).  16 MMAs of K 32.  The rope part is bf16: 4 kind::f16 MMAs
//                 (N = 16) into a second accumulator.
//   O^T += V^T P^T  M = 128 dims per block (4 blocks), N = 32, K = 128 tokens: A = the same
//                 codes read MN-major, B = the weights as e4m3 hi and lo rows per head.
//
// A softmax thread owns one token (one TMEM lane) and all 16 heads, so the scores need
// no cross-thread reduction; the running maxima only move when some thread votes for it
// (a named barrier with a predicate OR).  With x_t the scaled score and s_t the token's
// scale, the value logit is y_t = x_t log2(e) + log2(s_t), and the P operand is
// 2^(y_t - m_y + 4) for a lazy running maximum m_y of y (moved only by more than 4), which
// keeps it within (0, 256] -- e4m3 holds up to 448 -- and splits it into hi + lo codes
// (8 significant bits, like bf16).  The row sums use p_t = 2^(x_t log2(e) - m_x) with
// their own lazy maximum m_x (moved by more than 8).  At the end
//     out = 2^(m_y - 4 - m_x) (O_hi + O_lo) / l.
//
// Roles (384 threads): warp 0 streams each 128-token tile as five 16 KB ring slots (four
// code chunks of 128 dims, then kpe) plus the tile's scales with TMA; warp 1 allocates TMEM
// and one of its threads issues the MMAs (the scores of tile i + 1 go out before the values
// of tile i, within a segment); two softmax warpgroups (warps 4-7: heads 0-7, warps 8-11:
// heads 8-15) each take their heads of every token, and together set up each segment's
// query and write its output.  A split request's pieces write partials; the last CTA to
// finish one merges them in slot order (FlashMLA PR #233, "deterministic combine").  Every
// wait is bounded.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "attn.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace mla {

struct E4m3Cfg {
    static constexpr int kThreads = 384;
    static constexpr int kTile = kTileTokens;        // 128 tokens
    static constexpr int kSlotBytes = 128 * 128;     // 128 rows x 128 B: one code chunk or the kpe rows
    static constexpr int kSlots = 12;                // 5 per tile
    static constexpr int kScaleBufs = 4;             // per-tile scale buffers
    // a tile's scales, one box per page: page b of the tile at float offset b * max(P, 32) (a
    // tensor copy lands on a 128-byte boundary), 256 floats per buffer for every page size
    static constexpr int kScaleBufFloats = 256;
    static constexpr int kOffRing = 0;
    static constexpr int kOffQ = kOffRing + kSlots * kSlotBytes;   // [4 chunks][32 rows][128 B]: qh rows 0-15, ql 16-31
    static constexpr int kOffQpe = kOffQ + 4 * 32 * 128;           // [16 rows][128 B] bf16
    static constexpr int kOffP = kOffQpe + 16 * 128;               // 2 x [32 rows][128 B]: P hi rows 0-15, lo 16-31
    static constexpr int kPBytes = 32 * 128;
    static constexpr int kOffScale = kOffP + 2 * kPBytes;
    static constexpr int kOffMisc = kOffScale + kScaleBufs * kScaleBufFloats * 4;
    static constexpr int kMiscBytes = 2048;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kOffQ % 1024 == 0 && kOffQpe % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms");
    // TMEM columns: S buffers (scores 32 + rope 16) at 0 and 64, O^T blocks at 128 + 32 c
    static constexpr uint32_t kTmemCols = 256;
    static constexpr uint32_t kTmemO = 128;
    static constexpr uint32_t kIdescS = idesc_e4m3(128, 32, false, false);
    static constexpr uint32_t kIdescR = idesc_bf16(128, 16, false, false);
    static constexpr uint32_t kIdescO = idesc_e4m3(128, 32, true, false);
    // value logits: the running maximum moves only when a tile exceeds it by more than kYMove, and
    // the P operand is 2^(y - m_y + kPOffset) <= 2^(kYMove + kPOffset) = 256 (e4m3 holds 448)
    static constexpr float kYMove = 4.f;
    static constexpr float kPOffset = 4.f;
};

struct E4m3Misc {
    uint64_t full[E4m3Cfg::kSlots], empty[E4m3Cfg::kSlots];
    uint64_t sc_full[E4m3Cfg::kScaleBufs];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full[2], p_empty[2];
    uint64_t q_full, q_empty, drain;
    uint32_t tmem_base;
    int abort_flag;
    int merge_flag;
    float inv_sig[16];
    float red[2][2][4][8];   // [group][scores, value logits][warp][head]: tile maxima (rare path)
    float lsum[2][4][8];     // [group][warp][head]: row sums at a segment end
    float mrg_max[16], mrg_inv[16], mrg_w[128];
};

// D[tmem] (+)= A[smem] * B[smem]^T, e4m3 inputs, fp32 accumulate, issued by one thread.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two floats -> two e4m3 codes (the first in the lower byte), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3_pack2(float lo, float hi) {
    return __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// Two e4m3 codes (16 bits, lower byte first) -> their values (exact).
__device__ __forceinline__ float2 e4m3_unpack2(uint32_t codes) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(codes & 0xffffu)));
    return __half22float2(*reinterpret_cast<__half2*>(&r));
}

// x = hi + lo as e4m3 codes (two values at once, 16-bit code pairs): hi = e4m3(x),
// lo = e4m3(x - hi).  Exact when x has at most 8 significant bits and x - hi is not below the
// e4m3 subnormal range; otherwise lo carries the residual to 4 bits.
__device__ __forceinline__ void e4m3_split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = e4m3_pack2(x0, x1);
    const float2 h = e4m3_unpack2(hi);
    lo = e4m3_pack2(x0 - h.x, x1 - h.y);
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void st_shared_u8(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Byte offset of (row, byte) in a tile of 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_byte(uint32_t row, uint32_t byte) {
    return row * 128u + ((((byte >> 4) ^ (row & 7u))) << 4) + (byte & 15u);
}

// Debug timeline (-DMLA_TRACE): CTA 0 records the global timer at event `ev` (< 16) of tile
// `idx` (< 256) into prm.trace[ev * 256 + idx].
#ifdef MLA_TRACE
#define E4_TRACE(ev, idx)                                                                     \
    do {                                                                                      \
        if (prm.trace && blockIdx.x == 0 && (idx) < 256) prm.trace[(ev) * 256 + (idx)] = global_timer_ns(); \
    } while (0)
#else
#define E4_TRACE(ev, idx) \
    do {                  \
    } while (0)
#endif

__global__ void __launch_bounds__(E4m3Cfg::kThreads, 1)
    mla_decode_e4m3_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_kpe,
                           const __grid_constant__ CUtensorMap tm_scale, const AttnParams prm,
                           const uint16_t* __restrict__ q_nope, const uint16_t* __restrict__ q_pe) {
    using C = E4m3Cfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    E4m3Misc* misc = reinterpret_cast<E4m3Misc*>(smem + C::kOffMisc);
    static_assert(sizeof(E4m3Misc) <= C::kMiscBytes, "misc region");

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int unit = blockIdx.x / prm.head_groups;
    const int group_cta = blockIdx.x % prm.head_groups;
    const int head0 = group_cta * 16;
    const int seg_begin = prm.unit_ptr[unit];
    const int seg_end = prm.unit_ptr[unit + 1];
    const int P = prm.page_size;

    // Prologue before the previous kernel in the stream has finished (programmatic dependent
    // launch): barriers, TMEM and this CTA's slice of the plan, which only the plan commit
    // writes.  Every read of the caller's buffers and every write comes after grid_dep_wait.
    grid_dep_launch();
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(&misc->full[i], 1);
            mbar_init(&misc->empty[i], 1);
        }
        for (int i = 0; i < C::kScaleBufs; ++i) mbar_init(&misc->sc_full[i], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&misc->s_full[i], 1);
            mbar_init(&misc->s_empty[i], 8);   // one arrival per softmax warp
            mbar_init(&misc->p_full[i], 8);
            mbar_init(&misc->p_empty[i], 1);
        }
        mbar_init(&misc->q_full, 1);
        mbar_init(&misc->q_empty, 1);
        mbar_init(&misc->drain, 1);
        misc->abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&misc->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    grid_dep_wait();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;
    int* abort_flag = &misc->abort_flag;
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(abort_flag) != 0; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tm_codes);
            prefetch_tensormap(&tm_kpe);
            prefetch_tensormap(&tm_scale);
        }
        uint32_t kcount = 0, tcount = 0;
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
            const int nbox = (ntok + P - 1) / P;
            const int first_page = cur.t0 / P;
            const int seg_last_page = (cur.sg.t_end - 1) / P;
            if (first_page + nbox > win_base + 32 || first_page < win_base) {
                win_base = first_page;
                win_page = (win_base + lane <= seg_last_page) ? pages[win_base + lane] : 0;
            }
            for (int c = 0; c < 5 && ok; ++c) {   // code chunks of 128 dims, then kpe (with the scales)
                const uint32_t s = kcount % C::kSlots, use = kcount / C::kSlots;
                if (lane == 0 && use > 0) ok = wait_phase_flag(&misc->empty[s], (use - 1) & 1, abort_flag, prm.status, 61);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                if (lane == 0 && c == 0) E4_TRACE(0, tcount);
                uint8_t* dst = smem + C::kOffRing + s * C::kSlotBytes;
                // The tile's scales go to buffer tcount % 4.  Its previous tile (4 back) has been read:
                // this kpe slot's previous use was a code slot of the tile 2 back, released by that
                // tile's value MMAs, which follow its softmax, which follows the softmax 4 back.
                const uint32_t sb = tcount % C::kScaleBufs;
                float* sdst = reinterpret_cast<float*>(smem + C::kOffScale) + sb * C::kScaleBufFloats;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&misc->full[s], static_cast<uint32_t>(nbox * P * 128));
                    if (c == 4) mbar_arrive_expect_tx(&misc->sc_full[sb], static_cast<uint32_t>(nbox * P * 4));
                }
                for (int bx = 0; bx < nbox; ++bx) {
                    const int pg = __shfl_sync(0xffffffffu, win_page, (first_page + bx - win_base) & 31);
                    if (lane == 0) {
                        if (c < 4) {
                            tma_load_2d(dst + bx * P * 128, &tm_codes, &misc->full[s], c * 128, pg * P);
                        } else {
                            tma_load_2d(dst + bx * P * 128, &tm_kpe, &misc->full[s], 0, pg * P);
                            tma_load_1d(sdst + bx * (P < 32 ? 32 : P), &tm_scale, &misc->sc_full[sb], pg * P);
                        }
                    }
                }
                ++kcount;
            }
            if (lane == 0) E4_TRACE(5, tcount);
            ++tcount;
            more = cur.advance(new_seg);
        }
        if (lane == 0) {   // every copy lands before the CTA can exit
            const uint64_t t0 = global_timer_ns();
            for (int s = 0; s < C::kSlots; ++s) {
                const uint32_t uses = kcount / C::kSlots + (static_cast<uint32_t>(s) < kcount % C::kSlots ? 1 : 0);
                if (uses == 0) continue;
                while (!mbar_try_wait(&misc->full[s], (uses - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
            }
            for (int b = 0; b < C::kScaleBufs; ++b) {
                const uint32_t uses = tcount / C::kScaleBufs + (static_cast<uint32_t>(b) < tcount % C::kScaleBufs ? 1 : 0);
                if (uses == 0) continue;
                while (!mbar_try_wait(&misc->sc_full[b], (uses - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Per tile: the scores, then the values of the previous tile of the segment (the values of
        // a segment's last tile follow its scores at once).  The tensor pipe runs in issue order,
        // so the next tile's scores are done by the time its softmax starts.  (Issuing the values
        // as soon as P is ready, or filling waits with them, measured slower: the scores then
        // queue behind them and the softmax starts later.)
        if (lane == 0) {
            // descriptors built once; a byte offset advances the start-address field by offset / 16
            const uint64_t d_ring = umma_desc_sw128_c<16, 1024>(smem_u32(smem + C::kOffRing));
            const uint64_t d_ring_mn = umma_desc_sw128_c<C::kSlotBytes, 1024>(smem_u32(smem + C::kOffRing));
            const uint64_t d_q = umma_desc_sw128_c<16, 1024>(smem_u32(smem + C::kOffQ));
            const uint64_t d_qpe = umma_desc_sw128_c<16, 1024>(smem_u32(smem + C::kOffQpe));
            const uint64_t d_p = umma_desc_sw128_c<16, 1024>(smem_u32(smem + C::kOffP));
            uint32_t tcount = 0, kcount = 0, segc = 0;
            bool ok = true;
            // values of one tile: O^T[c] += V^T P^T over its 4 code slots (K = 128 tokens)
            auto issue_pv = [&](uint32_t tile, uint32_t kbase, bool first) {
                const uint32_t pb = tile & 1;
                ok = wait_phase_flag(&misc->p_full[pb], (tile >> 1) & 1, abort_flag, prm.status, 62);
                if (!ok) return;
                E4_TRACE(2, tile);
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const uint32_t s = (kbase + c) % C::kSlots;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_e4m3(tmem + C::kTmemO + 32 * c, d_ring_mn + ((s * C::kSlotBytes + k * 4096) >> 4),
                                  d_p + ((pb * C::kPBytes + k * 32) >> 4), C::kIdescO, (first && k == 0) ? 0u : 1u);
                    umma_commit(&misc->empty[s]);
                }
                umma_commit(&misc->p_empty[pb]);
            };
            bool pend = false, pend_first = false;
            uint32_t pend_tile = 0, pend_k = 0;
            TileCursorT<C::kTile> cur;
            bool more = cur.init(prm.segments, seg_begin, seg_end);
            bool new_seg = true;
            while (more && ok) {
                const bool last = cur.last();
                const bool first = cur.first();
                if (new_seg) {
                    ok = wait_phase_flag(&misc->q_full, segc & 1, abort_flag, prm.status, 63);
                    ++segc;
                }
                const uint32_t buf = tcount & 1;
                if (ok && tcount >= 2)
                    ok = wait_phase_flag(&misc->s_empty[buf], ((tcount >> 1) - 1) & 1, abort_flag, prm.status, 64);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + 64 * buf;
                for (int c = 0; c < 5 && ok; ++c) {
                    const uint32_t s = (kcount + c) % C::kSlots;
                    ok = wait_phase_flag(&misc->full[s], ((kcount + c) / C::kSlots) & 1, abort_flag, prm.status, 65);
                    if (!ok) break;
                    if (c == 0) E4_TRACE(6, tcount);
                    tc_fence_after();
                    const uint64_t a = d_ring + ((s * C::kSlotBytes) >> 4);
                    if (c < 4) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_e4m3(d, a + ((k * 32) >> 4), d_q + ((c * 4096 + k * 32) >> 4), C::kIdescS, (c | k) != 0);
                    } else {
                        E4_TRACE(1, tcount);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_bf16(d + 32, a + ((k * 32) >> 4), d_qpe + ((k * 32) >> 4), C::kIdescR, k != 0);
                        umma_commit(&misc->empty[s]);   // the kpe slot is done
                    }
                }
                if (!ok) break;
                umma_commit(&misc->s_full[buf]);
                if (last) umma_commit(&misc->q_empty);
                if (pend) {
                    issue_pv(pend_tile, pend_k, pend_first);
                    pend = false;
                }
                if (!ok) break;
                if (last) {
                    issue_pv(tcount, kcount, first);
                } else {
                    pend = true;
                    pend_tile = tcount;
                    pend_k = kcount;
                    pend_first = first;
                }
                kcount += 5;
                ++tcount;
                more = cur.advance(new_seg);
            }
            // drain: every MMA issued has completed before TMEM is released
            umma_commit(&misc->drain);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&misc->drain, 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
        }
#ifdef MLA_TRACE
    } else if (warp == 2) {
        // ------------------------------------------------------------ observer (trace builds only):
        // completion times of each tile's scores (10) and values (11); bounded by the wait limit
        if (lane == 0 && blockIdx.x == 0 && prm.trace) {
            TileCursorT<C::kTile> cur;
            bool more = cur.init(prm.segments, seg_begin, seg_end);
            bool new_seg = true;
            const uint64_t t0 = global_timer_ns();
            for (uint32_t j = 0; more && j < 256; ++j) {
                while (!mbar_test_wait(&misc->s_full[j & 1], (j >> 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
                E4_TRACE(10, j);
                while (!mbar_test_wait(&misc->p_empty[j & 1], (j >> 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
                E4_TRACE(11, j);
                more = cur.advance(new_seg);
            }
        }
#endif
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax groups, query set-up, epilogue
        const int grp = (warp - 4) / 4;                   // heads 8 grp .. 8 grp + 7
        const int t = (threadIdx.x - 128) % 128;          // token row / TMEM lane / dim row
        const int tid = threadIdx.x - 128;                // 0..255 over both groups
        const int hb = 8 * grp;
        const uint32_t lane_base = static_cast<uint32_t>(warp % 4) * 32;
        const uint32_t qb = smem_u32(smem + C::kOffQ);
        const uint32_t qpe = smem_u32(smem + C::kOffQpe);
        const uint32_t pbase = smem_u32(smem + C::kOffP);
        const float* scale_buf = reinterpret_cast<const float*>(smem + C::kOffScale);
        const uint32_t gbar = 1 + grp;   // this group's 128 threads
        const uint32_t abar = 3;         // both groups
        uint32_t tcount = 0, kcount = 0, segc = 0;
        bool ok = true;
        for (int si = seg_begin; si < seg_end && ok; ++si) {
            const Segment sg = prm.segments[si];
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
            if (sg.t_end <= sg.t_begin) {   // a request with no tokens
                for (int i = tid; i < 16 * kDimCkv; i += 256) st_out(od, o0 + i, 0.f);
                if (tid < 16) lbase[tid] = -INFINITY;
                continue;
            }
            // ---- query of this segment: thread (h = tid / 16, j = tid % 16) takes dims [32 j, 32 j + 32)
            if (segc > 0) ok = wait_phase_flag(&misc->q_empty, (segc - 1) & 1, abort_flag, prm.status, 66);
            ok = !named_barrier_or(abar, 256, !ok || aborted());
            if (!ok) break;
            {
                const int h = tid >> 4, j = tid & 15;
                const uint4* src = reinterpret_cast<const uint4*>(
                    q_nope + (static_cast<size_t>(sg.b) * prm.h_q + head0 + h) * kDimCkv + 32 * j);
                uint4 v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = src[i];
                float mx = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xffff0000u))));
                }
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                // sigma = 2^(7 - floor(log2 max)); a zero (or subnormal) row takes 2^7
                int e2 = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127;
                e2 = e2 < -100 ? 0 : (e2 > 100 ? 100 : e2);
                const float sig = __uint_as_float(static_cast<uint32_t>(127 + 7 - e2) << 23);
                if (j == 0) misc->inv_sig[h] = __uint_as_float(static_cast<uint32_t>(127 - 7 + e2) << 23);
                // 32 dims = 2 units of 16 bytes in chunk j / 4, units (j % 4) * 2, + 1
                const uint32_t chunk = qb + (j >> 2) * 4096;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint4 a = v[2 * u + q];
                        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            uint32_t h0, l0, h1, l1;
                            e4m3_split2(__uint_as_float(w[2 * e] << 16) * sig, __uint_as_float(w[2 * e] & 0xffff0000u) * sig,
                                        h0, l0);
                            e4m3_split2(__uint_as_float(w[2 * e + 1] << 16) * sig,
                                        __uint_as_float(w[2 * e + 1] & 0xffff0000u) * sig, h1, l1);
                            hw[2 * q + e] = h0 | (h1 << 16);
                            lw[2 * q + e] = l0 | (l1 << 16);
                        }
                    }
                    const uint32_t unit16 = (j & 3) * 2 + u;
                    st_shared_v4(chunk + h * 128 + ((unit16 ^ (h & 7)) << 4), hw[0], hw[1], hw[2], hw[3]);
                    st_shared_v4(chunk + (16 + h) * 128 + ((unit16 ^ ((16 + h) & 7)) << 4), lw[0], lw[1], lw[2], lw[3]);
                }
                if (tid < 128) {   // q_pe: 16 bytes (8 dims) of row tid / 8
                    const int hr = tid >> 3, jr = tid & 7;
                    const uint4 pe = *reinterpret_cast<const uint4*>(
                        q_pe + (static_cast<size_t>(sg.b) * prm.h_q + head0 + hr) * kDimKpe + 8 * jr);
                    st_shared_v4(qpe + hr * 128 + ((jr ^ (hr & 7)) << 4), pe.x, pe.y, pe.z, pe.w);
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(abar, 256);
            if (tid == 0) mbar_arrive(&misc->q_full);
            ++segc;
            float inv_sig[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) inv_sig[h] = misc->inv_sig[hb + h];
            float m_x[8], m_y[8], l[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                m_x[h] = -INFINITY;
                m_y[h] = -INFINITY;
                l[h] = 0.f;
            }
            bool first = true;
            for (int t0 = sg.t_begin; t0 < sg.t_end && ok; t0 += C::kTile) {
                const int ntok = min(C::kTile, sg.t_end - t0);
                const uint32_t buf = tcount & 1;
                const uint32_t sb = tcount % C::kScaleBufs;
                ok = wait_phase_flag(&misc->s_full[buf], (tcount >> 1) & 1, abort_flag, prm.status, 67);
                if (ok) ok = wait_phase_flag(&misc->sc_full[sb], (tcount / C::kScaleBufs) & 1, abort_flag, prm.status, 71);
                ok = !named_barrier_or(gbar, 128, !ok || aborted());
                if (!ok) break;
                if (t == 0) E4_TRACE(3 + 5 * grp, tcount);
                tc_fence_after();
                const bool valid = t < ntok;
                const float scale = valid ? scale_buf[sb * C::kScaleBufFloats + (t / P) * (P < 32 ? 32 : P) + t % P] : 0.f;
                float x[8];
                {
                    uint32_t rh[8], rl[8], rp[8];
                    tmem_ld8(tmem_addr(tmem, lane_base, 64 * buf + hb), rh);
                    tmem_ld8(tmem_addr(tmem, lane_base, 64 * buf + 16 + hb), rl);
                    tmem_ld8(tmem_addr(tmem, lane_base, 64 * buf + 32 + hb), rp);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const float lat = __uint_as_float(rh[h]) + __uint_as_float(rl[h]);
                        x[h] = valid ? fmaf(lat, inv_sig[h] * scale, __uint_as_float(rp[h])) * prm.scale_log2 : -INFINITY;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&misc->s_empty[buf]);
                // x holds the scores in log2 units; the value logits add log2(scale)
                const float ls = lg2_approx(scale);   // -inf for a zero scale or past the tile
                bool vote = false;
#pragma unroll
                for (int h = 0; h < 8; ++h) vote |= (x[h] > m_x[h] + 8.f) || (x[h] + ls > m_y[h] + C::kYMove);
                if (named_barrier_or(gbar, 128, vote)) {
                    // some running maximum moves: this group's head maxima of the tile
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const float wx = warp_max(x[h]);
                        const float wy = warp_max(x[h] + ls);
                        if (lane == 0) {
                            misc->red[grp][0][warp % 4][h] = wx;
                            misc->red[grp][1][warp % 4][h] = wy;
                        }
                    }
                    named_barrier_sync(gbar, 128);
                    float alpha_o[8];
                    bool resc = false;
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const float tx = fmaxf(fmaxf(misc->red[grp][0][0][h], misc->red[grp][0][1][h]),
                                               fmaxf(misc->red[grp][0][2][h], misc->red[grp][0][3][h]));
                        const float ty = fmaxf(fmaxf(misc->red[grp][1][0][h], misc->red[grp][1][1][h]),
                                               fmaxf(misc->red[grp][1][2][h], misc->red[grp][1][3][h]));
                        if (tx > m_x[h] + 8.f) {
                            l[h] *= fast_exp2(m_x[h] - tx);   // 0 when m_x was -inf
                            m_x[h] = tx;
                        }
                        alpha_o[h] = 1.f;
                        if (ty > m_y[h] + C::kYMove) {
                            alpha_o[h] = fast_exp2(m_y[h] - ty);
                            m_y[h] = ty;
                            resc = true;
                        }
                    }
                    named_barrier_sync(gbar, 128);   // red is rewritten by the next vote
                    if (resc && !first) {
                        // rescale this group's O^T columns (hi and lo of its heads) once the previous
                        // tile's values are in: its P buffer's release marks their completion
                        const uint32_t pt = tcount - 1;
                        ok = wait_phase_flag(&misc->p_empty[pt & 1], (pt >> 1) & 1, abort_flag, prm.status, 68);
                        ok = !named_barrier_or(gbar, 128, !ok);   // leave together or not at all
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
#pragma unroll
                            for (int part = 0; part < 2; ++part) {
                                uint32_t r[8];
                                const uint32_t addr = tmem_addr(tmem, lane_base, C::kTmemO + 32 * c + 16 * part + hb);
                                tmem_ld8(addr, r);
                                tmem_wait_ld();
#pragma unroll
                                for (int n = 0; n < 8; ++n) r[n] = __float_as_uint(__uint_as_float(r[n]) * alpha_o[n]);
                                tmem_st8(addr, r);
                            }
                        }
                        tmem_wait_st();
                        tc_fence_before();
                    }
                }
                // ---- P operand: hi and lo codes of 2^(y - m_y + 4) into column t of the P tile
                const uint32_t pb = tcount & 1;
                if (tcount >= 2) {
                    ok = wait_phase_flag(&misc->p_empty[pb], ((tcount >> 1) - 1) & 1, abort_flag, prm.status, 69);
                    ok = !named_barrier_or(gbar, 128, !ok);
                }
                if (!ok) break;
                const uint32_t pt_base = pbase + pb * C::kPBytes;
#pragma unroll
                for (int h = 0; h < 8; h += 2) {
                    l[h] += fast_exp2(x[h] - m_x[h]);
                    l[h + 1] += fast_exp2(x[h + 1] - m_x[h + 1]);
                    const float b0 = m_y[h] == -INFINITY ? 0.f : m_y[h] - C::kPOffset;
                    const float b1 = m_y[h + 1] == -INFINITY ? 0.f : m_y[h + 1] - C::kPOffset;
                    uint32_t hi, lo;
                    e4m3_split2(fast_exp2(x[h] + ls - b0), fast_exp2(x[h + 1] + ls - b1), hi, lo);
                    st_shared_u8(pt_base + sw128_byte(hb + h, t), hi & 0xffu);
                    st_shared_u8(pt_base + sw128_byte(hb + h + 1, t), (hi >> 8) & 0xffu);
                    st_shared_u8(pt_base + sw128_byte(16 + hb + h, t), lo & 0xffu);
                    st_shared_u8(pt_base + sw128_byte(17 + hb + h, t), (lo >> 8) & 0xffu);
                }
                if (ntok < C::kTile && t >= ntok) {
                    // value rows past the last token may hold anything (NaN codes included) and the
                    // value MMAs read all 128: zero this row in the tile's code slots (2 per group)
#pragma unroll
                    for (int c = 2 * grp; c < 2 * grp + 2; ++c) {
                        const uint32_t s = (kcount + c) % C::kSlots;
                        const uint32_t row = smem_u32(smem + C::kOffRing + s * C::kSlotBytes) + t * 128;
#pragma unroll
                        for (int u = 0; u < 8; ++u) st_shared_v4(row + 16 * u, 0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&misc->p_full[pb]);
                if (t == 0) E4_TRACE(4 + 5 * grp, tcount);
                first = false;
                kcount += 5;
                ++tcount;
            }
            if (!ok) break;
            // ---- epilogue: row sums over the group's 128 threads, then
            //      out = 2^(m_y - 4 - m_x) (O_hi + O_lo) / l for the group's 8 heads
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const float sm = warp_sum(l[h]);
                if (lane == 0) misc->lsum[grp][warp % 4][h] = sm;
            }
            {
                const uint32_t pt = tcount - 1;   // the segment's last tile
                ok = wait_phase_flag(&misc->p_empty[pt & 1], (pt >> 1) & 1, abort_flag, prm.status, 70);
            }
            ok = !named_barrier_or(gbar, 128, !ok || aborted()) && ok;
            if (!ok) break;
            tc_fence_after();
            float f[8], lt[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                lt[h] = (misc->lsum[grp][0][h] + misc->lsum[grp][1][h]) + (misc->lsum[grp][2][h] + misc->lsum[grp][3][h]);
                f[h] = (m_y[h] == -INFINITY || lt[h] == 0.f) ? 0.f : exp2f(m_y[h] - C::kPOffset - m_x[h]) / lt[h];
            }
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t rh[8], rl[8];
                tmem_ld8(tmem_addr(tmem, lane_base, C::kTmemO + 32 * c + hb), rh);
                tmem_ld8(tmem_addr(tmem, lane_base, C::kTmemO + 32 * c + 16 + hb), rl);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    st_out(od, o0 + static_cast<size_t>(hb + h) * kDimCkv + 128 * c + t,
                           (__uint_as_float(rh[h]) + __uint_as_float(rl[h])) * f[h]);
            }
            tc_fence_before();
            {
                // thread t < 8 of the group writes head hb + t's lse (a static select keeps the
                // arrays in registers)
                float mt = 0.f, ltt = 0.f;
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if (h == t) {
                        mt = m_x[h];
                        ltt = lt[h];
                    }
                if (t < 8) lbase[hb + t] = ltt > 0.f ? (mt + log2f(ltt)) * 0.69314718055994530942f : -INFINITY;
            }
            if (sg.slot >= 0) {
                // ---- split request: the last piece to arrive merges all of them in slot order,
                // both groups together (256 threads: one round of loads)
                __threadfence();
                named_barrier_sync(abar, 256);
                const int ctr = sg.item * prm.head_groups + group_cta;
                if (grp == 0 && t == 0) {
                    const int old = atomicAdd(&prm.counters[ctr], 1);
                    misc->merge_flag = (old == sg.n_slots - 1);
                }
                named_barrier_sync(abar, 256);
                if (misc->merge_flag) {
                    __threadfence();
                    merge_split_pieces_wide16(prm, sg.b, sg.slot_begin, sg.n_slots, head0, grp * 128 + t, abar, gbar,
                                              misc->mrg_max, misc->mrg_inv, misc->mrg_w);
                    if (grp == 0 && t == 0) prm.counters[ctr] = 0;
                }
                named_barrier_sync(abar, 256);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace mla
