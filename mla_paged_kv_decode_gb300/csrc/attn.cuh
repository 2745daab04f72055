// MLA paged decode attention kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// Absorbed MLA decode is MQA with one KV head: key [ckv | kpe] (576), value
// ckv (512) ("Benchmarking MLA", FlashInfer issue #700).  Each CTA owns HG query
// heads of every (request, token range) segment in its slot of the plan and
// walks the segment in 128-token tiles.  The two contractions are computed
// transposed, so that the token axis fills the 128-row UMMA M dimension even
// for 16 heads:
//
//   S^T[t, h]  = sum_k K[t, k] * Q[h, k]          (M = 128 tokens, N = HG, K = 576)
//   O^T[d, h] += sum_t V[t, d] * P[h, t]          (M = 128 dims x 4, N = HG, K = 128 tokens)
//
// with V = ckv read from the same shared-memory tile as K (the MN-major view of
// the K-major ckv rows).  Accumulators live in TMEM: S^T in HG columns and
// O^T in 4*HG columns, lane = token (S) or latent dim (O).
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q^T once per segment, then per tile the kpe rows
//               and the ckv rows of every page in the tile, 64-dim chunks with
//               the 128-byte swizzle, into a ring of 32 KB "pair" slots
//               (two 64-dim chunks = one 128-dim M block of the PV MMA) and
//               16 KB kpe slots, each with full/empty mbarriers.
//   warp 1      TMEM allocation; one thread issues every tcgen05.mma.
//   warps 2..5  softmax + epilogue: thread i of the group owns TMEM lane i
//               (token i of the tile for S^T, latent dim i (+128c) for O^T).
//
// Online softmax (log2 domain) with a lazily updated running max: a head's
// max is only moved (and O^T and the partial row sums rescaled) when the tile
// max exceeds it by more than 8 (a factor 256), so rescaling is rare; the
// final normalisation uses the same stale max for O and l, which keeps the
// result exact up to rounding.  P is rounded to bf16 for the PV MMA.
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
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s per wait before giving up

struct AttnParams {
    const int32_t* unit_ptr;      // [num_units + 1]
    const Segment* segments;      // [num_segments]
    const int32_t* kv_indices;
    const int32_t* kv_indptr;
    float* out;                   // [B, h_q, 512]
    float* lse;                   // [B, h_q]
    float* part_o;                // [num_partials, h_q, 512]
    float* part_lse;              // [num_partials, h_q]
    uint32_t* status;
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
    static constexpr int kPairSlots = 5;
    static constexpr int kKpeSlots = (HG == 16) ? 2 : 1;
    static constexpr int kChunkBytes = kTileTokens * 128;      // 64 dims x 128 tokens bf16
    static constexpr int kPairBytes = 2 * kChunkBytes;
    static constexpr int kQChunkBytes = HG * 128;              // 64 dims x HG heads
    static constexpr int kQBytes = 9 * kQChunkBytes;
    static constexpr int kPChunkBytes = HG * 128;              // 64 tokens x HG heads
    static constexpr int kPBytes = 2 * kPChunkBytes;

    static constexpr int kOffPair = 0;
    static constexpr int kOffKpe = kOffPair + kPairSlots * kPairBytes;
    static constexpr int kOffQ = kOffKpe + kKpeSlots * kChunkBytes;
    static constexpr int kOffP = kOffQ + ((kQBytes + 1023) / 1024) * 1024;
    static constexpr int kOffMisc = kOffP + ((kPBytes + 1023) / 1024) * 1024;
    static constexpr int kMiscBytes = 2048;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment slack

    // TMEM columns: S^T at 0 (HG), O^T chunk c at 64 + c*HG
    static constexpr uint32_t kTmemS = 0;
    static constexpr uint32_t kTmemO = 64;
    static constexpr uint32_t kTmemCols = (64 + 4 * HG <= 128) ? 128 : 256;

    static constexpr uint32_t kIdescS = idesc_bf16(128, HG, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16(128, HG, true, false);
};

struct AttnMisc {
    uint64_t q_full, q_empty, s_full, p_full, o_full, drain;
    uint64_t kfull[2], kempty[2];
    uint64_t pfull[5], pempty[5];
    uint32_t tmem_base;
    int abort_flag;
    float red_max[2][4][32];
    float red_sum[4][32];
};

static_assert(sizeof(AttnMisc) <= 2048, "misc region");

// Bounded wait on an mbarrier phase.  Returns false if the kernel is aborting.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, AttnMisc* misc, uint32_t* status,
                                           uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int*>(&misc->abort_flag)) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *reinterpret_cast<volatile int*>(&misc->abort_flag) = 1;
            atomicCAS(status, 0u, kStatusTimeout | site);
            return false;
        }
    }
}

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
    uint8_t* q_smem = smem + C::kOffQ;
    uint8_t* p_smem = smem + C::kOffP;
    AttnMisc* misc = reinterpret_cast<AttnMisc*>(smem + C::kOffMisc);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int unit = blockIdx.x / prm.head_groups;
    const int group = blockIdx.x % prm.head_groups;
    const int seg_begin = prm.unit_ptr[unit];
    const int seg_end = prm.unit_ptr[unit + 1];
    const int P = prm.page_size;

    if (threadIdx.x == 0) {
        mbar_init(&misc->q_full, 1);
        mbar_init(&misc->q_empty, 1);
        mbar_init(&misc->s_full, 1);
        mbar_init(&misc->p_full, C::kSoftmaxThreads);
        mbar_init(&misc->o_full, 1);
        mbar_init(&misc->drain, 1);
        for (int i = 0; i < C::kKpeSlots; ++i) {
            mbar_init(&misc->kfull[i], 1);
            mbar_init(&misc->kempty[i], 1);
        }
        for (int i = 0; i < C::kPairSlots; ++i) {
            mbar_init(&misc->pfull[i], 1);
            mbar_init(&misc->pempty[i], 1);
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
        uint32_t kcount = 0, pcount = 0, nseg = 0;
        bool ok = true;
        for (int si = seg_begin; si < seg_end && ok; ++si, ++nseg) {
            const Segment sg = prm.segments[si];
            const int32_t* pages = prm.kv_indices + prm.kv_indptr[sg.b];
            if (lane == 0) {
                if (nseg > 0) ok = wait_phase(&misc->q_empty, (nseg - 1) & 1, misc, prm.status, 1);
                if (ok) {
                    mbar_arrive_expect_tx(&misc->q_full, C::kQBytes);
                    const int row = sg.b * prm.h_q + group * HG;
                    for (int c = 0; c < 8; ++c) tma_load_2d(q_smem + c * C::kQChunkBytes, &tm_qn, &misc->q_full, c * 64, row);
                    tma_load_2d(q_smem + 8 * C::kQChunkBytes, &tm_qp, &misc->q_full, 0, row);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            for (int t0 = sg.t_begin; t0 < sg.t_end && ok; t0 += kTileTokens) {
                const int ntok = min(kTileTokens, sg.t_end - t0);
                const int first_page = t0 / P;
                const int npages = (ntok + P - 1) / P;
                const int my_page = lane < npages ? pages[first_page + lane] : 0;
                const uint32_t bytes = static_cast<uint32_t>(npages * P * 128);
                // kpe rows of the tile
                {
                    const uint32_t s = kcount % C::kKpeSlots;
                    const uint32_t use = kcount / C::kKpeSlots;
                    if (lane == 0 && use > 0) ok = wait_phase(&misc->kempty[s], (use - 1) & 1, misc, prm.status, 2);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    if (lane == 0) mbar_arrive_expect_tx(&misc->kfull[s], bytes);
                    uint8_t* dst = kpe_base + s * C::kChunkBytes;
                    for (int i = 0; i < npages; ++i) {
                        const int pg = __shfl_sync(0xffffffffu, my_page, i);
                        if (lane == 0) tma_load_2d(dst + i * P * 128, &tm_kpe, &misc->kfull[s], 0, pg * P);
                    }
                    ++kcount;
                }
                // ckv rows, one pair slot per 128 latent dims
                for (int c = 0; c < 4 && ok; ++c) {
                    const uint32_t s = pcount % C::kPairSlots;
                    const uint32_t use = pcount / C::kPairSlots;
                    if (lane == 0 && use > 0) ok = wait_phase(&misc->pempty[s], (use - 1) & 1, misc, prm.status, 3);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok) break;
                    if (lane == 0) mbar_arrive_expect_tx(&misc->pfull[s], 2 * bytes);
                    uint8_t* dst = pair_base + s * C::kPairBytes;
                    for (int i = 0; i < npages; ++i) {
                        const int pg = __shfl_sync(0xffffffffu, my_page, i);
                        if (lane == 0) {
                            tma_load_2d(dst + i * P * 128, &tm_ckv, &misc->pfull[s], (2 * c) * 64, pg * P);
                            tma_load_2d(dst + C::kChunkBytes + i * P * 128, &tm_ckv, &misc->pfull[s], (2 * c + 1) * 64,
                                        pg * P);
                        }
                    }
                    ++pcount;
                }
            }
        }
        // teardown: let every copy this warp issued land before the CTA can exit
        if (lane == 0) {
            const uint64_t t0 = global_timer_ns();
            auto drain = [&](uint64_t* bar, uint32_t uses) {
                if (uses == 0) return;
                while (!mbar_try_wait(bar, (uses - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
            };
            drain(&misc->q_full, nseg);
            for (int s = 0; s < C::kKpeSlots; ++s)
                drain(&misc->kfull[s], kcount / C::kKpeSlots + (static_cast<uint32_t>(s) < kcount % C::kKpeSlots ? 1 : 0));
            for (int s = 0; s < C::kPairSlots; ++s)
                drain(&misc->pfull[s], pcount / C::kPairSlots + (static_cast<uint32_t>(s) < pcount % C::kPairSlots ? 1 : 0));
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t kcount = 0, pcount = 0, tcount = 0, nseg = 0;
            bool ok = true;
            const uint32_t q_addr = smem_u32(q_smem);
            const uint32_t p_addr = smem_u32(p_smem);
            for (int si = seg_begin; si < seg_end && ok; ++si, ++nseg) {
                const Segment sg = prm.segments[si];
                ok = wait_phase(&misc->q_full, nseg & 1, misc, prm.status, 4);
                for (int t0 = sg.t_begin; t0 < sg.t_end && ok; t0 += kTileTokens, ++tcount) {
                    const bool first_tile = (t0 == sg.t_begin);
                    const bool last_tile = (t0 + kTileTokens >= sg.t_end);
                    // ---- S^T = K Q^T : kpe part (q chunk 8), then the 8 ckv chunks
                    const uint32_t ks = kcount % C::kKpeSlots;
                    ok = wait_phase(&misc->kfull[ks], (kcount / C::kKpeSlots) & 1, misc, prm.status, 5);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kaddr = smem_u32(kpe_base + ks * C::kChunkBytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_bf16(tmem + C::kTmemS, umma_desc_sw128(kaddr + k * 32, 16, 1024),
                                  umma_desc_sw128(q_addr + 8 * C::kQChunkBytes + k * 32, 16, 1024), C::kIdescS,
                                  k > 0);
                    uint32_t pslot[4];
                    for (int c = 0; c < 4 && ok; ++c) {
                        pslot[c] = (pcount + c) % C::kPairSlots;
                        ok = wait_phase(&misc->pfull[pslot[c]], ((pcount + c) / C::kPairSlots) & 1, misc, prm.status, 6);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t paddr = smem_u32(pair_base + pslot[c] * C::kPairBytes);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                umma_bf16(tmem + C::kTmemS, umma_desc_sw128(paddr + h * C::kChunkBytes + k * 32, 16, 1024),
                                          umma_desc_sw128(q_addr + (2 * c + h) * C::kQChunkBytes + k * 32, 16, 1024),
                                          C::kIdescS, 1);
                    }
                    if (!ok) break;
                    umma_commit(&misc->kempty[ks]);
                    ++kcount;
                    if (last_tile) umma_commit(&misc->q_empty);
                    umma_commit(&misc->s_full);
                    // ---- O^T += V^T P^T once the softmax group has written P
                    ok = wait_phase(&misc->p_full, tcount & 1, misc, prm.status, 7);
                    if (!ok) break;
                    tc_fence_after();
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t paddr = smem_u32(pair_base + pslot[c] * C::kPairBytes);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_bf16(tmem + C::kTmemO + c * HG,
                                      umma_desc_sw128(paddr + kk * 2048, C::kChunkBytes, 1024),
                                      umma_desc_sw128(p_addr + (kk / 4) * C::kPChunkBytes + (kk % 4) * 32, 16, 1024),
                                      C::kIdescPV, (first_tile && kk == 0) ? 0u : 1u);
                        umma_commit(&misc->pempty[pslot[c]]);
                    }
                    pcount += 4;
                    if (last_tile) umma_commit(&misc->o_full);
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
        const int row = sp * 32 + lane;          // TMEM lane: token of the tile / latent dim
        const int gtid = threadIdx.x - 64;       // 0..127 within the group
        uint32_t tcount = 0, nseg = 0, pcount = 0;
        bool ok = true;
        for (int si = seg_begin; si < seg_end && ok; ++si, ++nseg) {
            const Segment sg = prm.segments[si];
            float m_run[HG], l_part[HG];
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                m_run[h] = -INFINITY;
                l_part[h] = 0.f;
            }
            for (int t0 = sg.t_begin; t0 < sg.t_end; t0 += kTileTokens, ++tcount, pcount += 4) {
                const bool first_tile = (t0 == sg.t_begin);
                const int ntok = min(kTileTokens, sg.t_end - t0);
                const bool valid = row < ntok;
                ok = wait_phase(&misc->s_full, tcount & 1, misc, prm.status, 8);
                const bool bad = named_barrier_or(1, C::kSoftmaxThreads,
                                                  !ok || *reinterpret_cast<volatile int*>(&misc->abort_flag));
                if (bad) { ok = false; break; }
                tc_fence_after();
                float x[HG];
#pragma unroll
                for (int j = 0; j < HG / 16; ++j) tmem_ld16(tmem_addr(tmem, sp * 32, C::kTmemS + 16 * j), x + 16 * j);
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
                // P^T[h][t] in bf16, K-major 128B-swizzled rows of 64 tokens
                {
                    uint8_t* pchunk = p_smem + (row >> 6) * C::kPChunkBytes;
                    const int col = row & 63;
#pragma unroll
                    for (int h = 0; h < HG; ++h) {
                        const float p = exp2f(x[h] - m_run[h]);
                        l_part[h] += p;
                        *reinterpret_cast<__nv_bfloat16*>(pchunk + sw128_offset(h, col)) = __float2bfloat16_rn(p);
                    }
                }
                if (!valid) {
                    // rows past the request's end may hold stale or NaN bytes: zero the value rows
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t s = (pcount + c) % C::kPairSlots;
                        uint4* r0 = reinterpret_cast<uint4*>(pair_base + s * C::kPairBytes + row * 128);
                        uint4* r1 = reinterpret_cast<uint4*>(pair_base + s * C::kPairBytes + C::kChunkBytes + row * 128);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            r0[i] = make_uint4(0, 0, 0, 0);
                            r1[i] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&misc->p_full);
            }
            if (!ok) break;
            // ---- epilogue: wait for the last PV, normalise, store
            ok = wait_phase(&misc->o_full, nseg & 1, misc, prm.status, 9);
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
            const size_t head0 = static_cast<size_t>(group) * HG;
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
                    for (int i = 0; i < 16; ++i) obase[static_cast<size_t>(16 * j + i) * kDimCkv + c * 128 + row] = o[i] * inv_l[16 * j + i];
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
            // red_sum is reused by the next segment only after its own barriers
            named_barrier_sync(1, C::kSoftmaxThreads);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace mla
