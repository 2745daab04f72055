// MLA paged decode attention over an INT8 latent cache (two's-complement codes with one fp32
// scale per token, bf16 kpe) for 16 or 32 query heads per CTA on sm_103a: TMA staging of the
// 8-bit stages, an in-CTA expansion of the codes to f16 tiles, and warp-level mma.sync
// (m16n8k16, f32 accumulate) on them.
//
// The cache holds token t's latent as ckv_t = s_t * code_t (FlashMLA PR #233, "FP8 e4m3 or
// INT8 with one scale per token (644 instead of 1152 bytes per token), dequantized inside the
// kernel").  Every INT8 code is exact in f16, so two warps of the producer warpgroup expand
// each stage's codes into an f16 tile in the layout of the bf16 narrow kernel
// (attn_narrow.cuh); the compute warps then run the same split-K score and P V contractions
// with f16 operands:
//
//   scores   x_t = sm_scale * (s_t * (q_nope . code_t) + q_pe . kpe_t).  The latent query of
//            head h enters as f16(q_nope * sigma_h), sigma_h a power of two that puts its
//            largest |q| in [2^14, 2^15); the product sums are exact in the MMA's fp32
//            accumulation and are rescaled by s_t / sigma_h.  The rope part stays bf16.
//   values   O += sum_t p_t (s_t / c) code_t with p_t the softmax weight (lazy running max, as
//            in the bf16 kernel) and c a lazy running maximum of the segment's token scales
//            (moved, and O rescaled, only when a tile's largest scale exceeds it by 16x), so
//            the f16 weights p_t s_t / c stay below 2^12.  At the end out = c O / l.
//
// Roles (384 threads): warps 0-1 issue the TMA copies of the stages (8-bit codes with the
// 128-byte swizzle, kpe, the token scales), warps 2-3 expand the codes, warps 4-11 are the
// compute groups of the bf16 kernel (two token groups taking alternate tiles for 16 heads,
// two head groups for 32).  A split request's pieces are merged as in the bf16 kernel: the
// piece with the last arrival ticket merges all of them in slot order (FlashMLA PR #233,
// "deterministic combine").  Every wait is bounded.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn.cuh"
#include "attn_narrow.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace mla {

template <int HG>
struct Narrow8Cfg {
    static_assert(HG == 16 || HG == 32, "heads per CTA");
    static constexpr int kHeadGroups = HG / 16;
    static constexpr int kTokenGroups = (HG == 16) ? 2 : 1;
    static constexpr int kGroups = kHeadGroups * kTokenGroups;
    static constexpr int kComputeWarps = 4 * kGroups;          // 8
    static constexpr int kProducerWarps = 4;                   // warps 0-1 issue, 2-3 expand
    static constexpr int kIssuers = 2;
    static constexpr int kConverters = 2;
    static constexpr int kThreads = 32 * (kProducerWarps + kComputeWarps);
    static constexpr uint32_t kProducerRegs = 88;
    static constexpr uint32_t kComputeRegs = 208;
    static_assert(128 * kProducerRegs + 32 * kComputeWarps * kComputeRegs <= 65536 / kThreads / 8 * 8 * kThreads,
                  "register split");
    // an 8-bit ring stage of 32 tokens: 4 code boxes [32 rows][128 B] (128-byte swizzle), the kpe
    // rows [32][128 B] (128-byte swizzle), the scales (page b of the stage at float 32 b)
    static constexpr int kCodeBoxBytes = 32 * 128;
    static constexpr int kKpeOff = 4 * kCodeBoxBytes;
    static constexpr int kScaleOff = kKpeOff + 32 * 128;
    static constexpr int kStageBytes = 21504;                  // 1024-aligned
    static_assert(kScaleOff + 256 <= kStageBytes, "stage layout");
    static constexpr int kStages = 5;
    // expanded f16 tiles: [8 chunks of 64 dims][32 rows][128 B], 128-byte swizzle
    static constexpr int kXChunkBytes = 32 * 128;
    static constexpr int kXBytes = 8 * kXChunkBytes;
    static constexpr int kXBufs = 3;                           // lets the expansion run ahead of the compute
    static constexpr int kPartBytes = 4 * 32 * 16 * 4;
    static constexpr int kPRowBytes = 80;
    static constexpr int kGroupScratch = 16 * kPRowBytes + 4 * 16 * 4;
    static constexpr int kOffStage = 0;
    static constexpr int kOffX = kOffStage + kStages * kStageBytes;
    static constexpr int kOffPart = kOffX + kXBufs * kXBytes;
    static constexpr int kOffScratch = kOffPart + kGroups * kPartBytes;
    static constexpr int kOffMisc = kOffScratch + kGroups * kGroupScratch;
    static constexpr int kMiscBytes = 3072;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;
    static_assert(kOffX % 1024 == 0, "swizzle atoms");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kTokenGroups == 1 || 2 * kGroups * kPartBytes >= 16 * kDimCkv * 4 / 2, "merge buffer");
};

struct Narrow8Misc {
    uint64_t full[5], empty[5];
    uint64_t xfull[3], xempty[3];
    int abort_flag;
    int merge_flag[2];
    float sig[2][16], isig[2][16];   // per head group: sigma_h and 1 / sigma_h of the segment's query
    float mrg_max[2][16];
    float mrg_inv[2][16];
    float mrg_w[2][128];
    float tg_m[16], tg_l[16];        // token-group merge: running max, row sum of group 1
    float tg_c;                      // ... and its running scale maximum
};

// Four INT8 codes (one 32-bit word, first code in the lowest byte) -> four f16 values, exactly:
// b + 128 as an unsigned byte u, placed under the f16 exponent of 1024 (0x64), reads 1024 + u;
// subtracting 1152 leaves b (f16 holds every integer below 2048).
__device__ __forceinline__ void expand4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t h01 = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t h23 = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 k = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6480)));   // 1152
    __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&h01), k);
    __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&h23), k);
    lo = *reinterpret_cast<uint32_t*>(&a);
    hi = *reinterpret_cast<uint32_t*>(&b);
}

template <int HG>
__global__ void __launch_bounds__(Narrow8Cfg<HG>::kThreads, 1)
    mla_decode_narrow8_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_kpe,
                              const __grid_constant__ CUtensorMap tm_scale, const AttnParams prm,
                              const uint16_t* __restrict__ q_nope, const uint16_t* __restrict__ q_pe) {
    using C = Narrow8Cfg<HG>;
    static_assert(sizeof(Narrow8Misc) <= C::kMiscBytes && C::kStages <= 5 && C::kXBufs <= 3, "misc region");
    constexpr int kTile = kNarrowTile;   // 32 tokens = one stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stage_base = smem + C::kOffStage;
    uint8_t* xbase = smem + C::kOffX;
    float* part_base = reinterpret_cast<float*>(smem + C::kOffPart);
    Narrow8Misc* misc = reinterpret_cast<Narrow8Misc*>(smem + C::kOffMisc);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int unit = blockIdx.x / prm.head_groups;
    const int group_cta = blockIdx.x % prm.head_groups;
    const int seg_begin = prm.unit_ptr[unit];
    const int seg_end = prm.unit_ptr[unit + 1];
    const int P = prm.page_size;
    const int box_rows = P < kTile ? P : kTile;

    // Prologue before the previous kernel in the stream has finished (programmatic dependent
    // launch): barriers and this CTA's slice of the plan.  Every read of the caller's buffers
    // and every write comes after grid_dep_wait.
    grid_dep_launch();
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&misc->full[i], 1);
            // released by the two expanding warps and the 4 warps of every 16-head group that
            // reads the stage's kpe and scales
            mbar_init(&misc->empty[i], C::kConverters + 4 * C::kHeadGroups);
        }
        for (int i = 0; i < C::kXBufs; ++i) {
            mbar_init(&misc->xfull[i], C::kConverters);
            mbar_init(&misc->xempty[i], 4 * C::kHeadGroups);
        }
        misc->abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_codes);
        prefetch_tensormap(&tm_kpe);
        prefetch_tensormap(&tm_scale);
    }
    __syncthreads();
    grid_dep_wait();

    if (warp < C::kProducerWarps) regs_dec<C::kProducerRegs>();
    else regs_inc<C::kComputeRegs>();

    if (warp < C::kIssuers) {
        // ------------------------------------------------------------ TMA producers (stage s % 2 == warp)
        const int pid = warp;
        uint32_t scount = 0;
        bool ok = true;
        TileCursorT<kTile> cur;
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
            const int nbox = (ntok + box_rows - 1) / box_rows;
            const int first_page = cur.t0 / P;
            const int last_page_st = (cur.t0 + nbox * box_rows - 1) / P;
            if (last_page_st + 1 > win_base + 32 || first_page < win_base) {
                const int seg_last_page = (cur.sg.t_end - 1) / P;
                win_base = first_page;
                win_page = (win_base + lane <= seg_last_page) ? pages[win_base + lane] : 0;
            }
            const uint32_t s = scount % C::kStages, use = scount / C::kStages;
            if (static_cast<int>(s) % C::kIssuers == pid) {
                if (lane == 0 && use > 0)
                    ok = wait_phase_flag(&misc->empty[s], (use - 1) & 1, &misc->abort_flag, prm.status, 31);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (ok) {
                    uint8_t* dst = stage_base + s * C::kStageBytes;
                    if (lane == 0) MLA_TRACE_EVENT(0, scount);
                    if (lane == 0)
                        mbar_arrive_expect_tx(&misc->full[s],
                                              static_cast<uint32_t>(nbox * box_rows * (kDimCkv + kDimKpe * 2 + 4)));
                    for (int bx = 0; bx < nbox; ++bx) {
                        const int t = cur.t0 + bx * box_rows;
                        const int pg = __shfl_sync(0xffffffffu, win_page, (t / P - win_base) & 31);
                        if (lane == 0) {
                            const int y = pg * P + (t % P);
                            for (int xb = 0; xb < 4; ++xb)
                                tma_load_2d(dst + xb * C::kCodeBoxBytes + bx * box_rows * 128, &tm_codes, &misc->full[s],
                                            xb * 128, y);
                            tma_load_2d(dst + C::kKpeOff + bx * box_rows * 128, &tm_kpe, &misc->full[s], 0, y);
                            tma_load_1d(dst + C::kScaleOff + bx * 128, &tm_scale, &misc->full[s], y);
                        }
                    }
                }
            }
            ++scount;
            more = cur.advance(new_seg);
        }
        if (lane == 0) {   // every copy of this producer's stages lands before the CTA can exit
            const uint64_t t0 = global_timer_ns();
            for (int s = pid; s < C::kStages; s += C::kIssuers) {
                const uint32_t uses = scount / C::kStages + (static_cast<uint32_t>(s) < scount % C::kStages ? 1 : 0);
                if (uses == 0) continue;
                while (!mbar_try_wait(&misc->full[s], (uses - 1) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
            }
        }
    } else if (warp < C::kProducerWarps) {
        // ------------------------------------------------------------ code expansion (warps 2, 3)
        // Tile t: ring stage t % kStages -> f16 tile t % 2.  The 32 blocks of a tile (4 row octets
        // x 8 chunks of 64 dims) alternate between the two warps; in a block lane (r, q) takes row
        // 8 o + r and the 16 codes of source unit 4 c + q, which become 16 f16 (2 swizzled units).
        const int cv = warp - C::kIssuers;   // 0, 1
        const int r8 = lane >> 2, q4 = lane & 3;
        uint32_t tcount = 0;
        bool ok = true;
        TileCursorT<kTile> cur;
        bool more = cur.init(prm.segments, seg_begin, seg_end);
        bool new_seg = true;
        while (more && ok) {
            const int ntok = cur.ntok();
            const uint32_t s = tcount % C::kStages, xb = tcount % C::kXBufs;
            if (lane == 0) {
                ok = wait_phase_flag(&misc->full[s], (tcount / C::kStages) & 1, &misc->abort_flag, prm.status, 32);
                if (ok && tcount >= C::kXBufs)
                    ok = wait_phase_flag(&misc->xempty[xb], (tcount / C::kXBufs - 1) & 1, &misc->abort_flag, prm.status,
                                         33);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            // every lane observes the completed phases itself (they are complete: no waiting)
            (void)mbar_try_wait(&misc->full[s], (tcount / C::kStages) & 1);
            if (tcount >= C::kXBufs) (void)mbar_try_wait(&misc->xempty[xb], (tcount / C::kXBufs - 1) & 1);
            const uint32_t src = smem_u32(stage_base + s * C::kStageBytes);
            const uint32_t dstb = smem_u32(xbase + xb * C::kXBytes);
            if (lane == 0 && cv == 0) MLA_TRACE_EVENT(1, tcount);
            // blocks cv, cv + 2, ..., 30 + cv, four at a time: their loads are in flight together
#pragma unroll
            for (int i0 = 0; i0 < 16; i0 += 4) {
                uint32_t c[4][4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int blk = cv + 2 * (i0 + k);
                    const int row = (blk & 3) * 8 + r8;
                    const int u = (blk >> 2) * 4 + q4;   // source unit of 16 codes
                    c[k][0] = c[k][1] = c[k][2] = c[k][3] = 0u;
                    if (row < ntok) {
                        const uint32_t a = src + (u >> 3) * C::kCodeBoxBytes + row * 128 + (((u & 7) ^ r8) << 4);
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(c[k][0]), "=r"(c[k][1]), "=r"(c[k][2]), "=r"(c[k][3])
                                     : "r"(a));
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int blk = cv + 2 * (i0 + k);
                    const int row = (blk & 3) * 8 + r8;
                    const uint32_t rowb = dstb + (blk >> 2) * C::kXChunkBytes + row * 128;
                    uint32_t w[8];
                    expand4(c[k][0], w[0], w[1]);
                    expand4(c[k][1], w[2], w[3]);
                    expand4(c[k][2], w[4], w[5]);
                    expand4(c[k][3], w[6], w[7]);
                    // codes 0 (rows past the last token) expand to +0
                    st_shared_v4(rowb + (((2 * q4) ^ r8) << 4), w[0], w[1], w[2], w[3]);
                    st_shared_v4(rowb + (((2 * q4 + 1) ^ r8) << 4), w[4], w[5], w[6], w[7]);
                }
            }
            __syncwarp();
            if (lane == 0 && cv == 0) MLA_TRACE_EVENT(6, tcount);
            if (lane == 0) {
                mbar_arrive(&misc->xfull[xb]);
                mbar_arrive(&misc->empty[s]);
            }
            ++tcount;
            more = cur.advance(new_seg);
        }
    } else {
        // ------------------------------------------------------------ compute warps
        const int cw = warp - C::kProducerWarps;
        const int grp = cw / 4;
        const int hgi = grp / C::kTokenGroups;
        const int tg = grp % C::kTokenGroups;
        const int kr = cw % 4;
        const int g = lane >> 2, c4 = lane & 3;
        const int gt = kr * 32 + lane;
        const uint32_t named_bar = 1 + grp;
        const uint32_t merge_bar = 1 + C::kGroups + hgi;
        const int head0 = group_cta * HG + hgi * 16;
        float* part = part_base + grp * (C::kPartBytes / 4);
        uint8_t* pbuf = smem + C::kOffScratch + grp * C::kGroupScratch;
        float* rowmax = reinterpret_cast<float*>(pbuf + 16 * C::kPRowBytes);
        uint32_t tcount = 0;   // tiles of the CTA so far (both token groups)
        bool ok = true;
        uint32_t qa[9][4];
        float isg[2];          // 1 / sigma of rows g and g + 8
        // sigma_h for the group's 16 heads: 8 threads a head, 64 latent dims each
        auto set_sigma = [&](int b) {
            const int hh = gt >> 3, sub = gt & 7;
            const uint4* qrow = reinterpret_cast<const uint4*>(q_nope + (static_cast<size_t>(b) * prm.h_q + head0 + hh) * kDimCkv) +
                                sub * 8;
            float mx = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 v = qrow[j];
                const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    mx = fmaxf(mx, fabsf(__uint_as_float(ws[e] << 16)));
                    mx = fmaxf(mx, fabsf(__uint_as_float(ws[e] & 0xffff0000u)));
                }
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            if (sub == 0) {
                // biased exponent of sigma: 141 - e(max) puts the largest |q| sigma in [2^14, 2^15)
                const int eb = static_cast<int>((__float_as_uint(mx) >> 23) & 0xff);
                int sb = 268 - eb;
                sb = sb < 1 ? 1 : (sb > 253 ? 253 : sb);   // sigma and 1 / sigma both normal
                const float sg_ = __uint_as_float(static_cast<uint32_t>(sb) << 23);
                misc->sig[hgi][hh] = sg_;
                misc->isig[hgi][hh] = __uint_as_float(static_cast<uint32_t>(254 - sb) << 23);   // 2^-(sb - 127)
            }
        };
        auto load_q = [&](int b) {
            const size_t qrow0 = static_cast<size_t>(b) * prm.h_q + head0;
            const float sg0 = misc->sig[hgi][g], sg1 = misc->sig[hgi][g + 8];
            isg[0] = misc->isig[hgi][g];
            isg[1] = misc->isig[hgi][g + 8];
#pragma unroll
            for (int ks = 0; ks < 9; ++ks) {
                const int kd = kr * 144 + ks * 16;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int row = g + ((r & 1) ? 8 : 0);
                    const int dim = kd + 2 * c4 + ((r & 2) ? 8 : 0);
                    if (dim < kDimCkv) {
                        const uint32_t v = *reinterpret_cast<const uint32_t*>(q_nope + (qrow0 + row) * kDimCkv + dim);
                        const float sgr = (r & 1) ? sg1 : sg0;
                        qa[ks][r] = pack_f16(__uint_as_float(v << 16) * sgr, __uint_as_float(v & 0xffff0000u) * sgr);
                    } else {
                        qa[ks][r] = *reinterpret_cast<const uint32_t*>(q_pe + (qrow0 + row) * kDimKpe + (dim - kDimCkv));
                    }
                }
            }
        };
        for (int si = seg_begin; si < seg_end && ok; ++si) {
            const Segment sg = prm.segments[si];
            if (sg.t_end <= sg.t_begin) {
                if (tg == 0) {
                    const size_t o0 = (static_cast<size_t>(sg.b) * prm.h_q + head0) * kDimCkv;
                    for (int i = gt; i < 16 * kDimCkv; i += 128) st_out(final_out(prm), o0 + i, 0.f);
                    if (kr == 0 && lane < 16) prm.lse[static_cast<size_t>(sg.b) * prm.h_q + head0 + lane] = -INFINITY;
                }
                continue;
            }
            // sigma of the segment's query (one token group computes it; both read it after the barrier)
            if (tg == 0) set_sigma(sg.b);
            if (C::kTokenGroups == 2) named_barrier_sync(merge_bar, 256);
            else named_barrier_sync(named_bar, 128);
            load_q(sg.b);
            float o[16][4];
#pragma unroll
            for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            float m_run[2] = {-INFINITY, -INFINITY};
            float l_part[2] = {0.f, 0.f};
            float c_run = 0.f;   // running maximum of the token scales (lazy)
            int tile_in_seg = 0;
            for (int t0 = sg.t_begin; t0 < sg.t_end; t0 += kTile, ++tile_in_seg, ++tcount) {
                const int ntok = min(kTile, sg.t_end - t0);
                if (tile_in_seg % C::kTokenGroups != tg) continue;   // the other token group's tile
                const uint32_t sl = tcount % C::kStages, xb = tcount % C::kXBufs;
                // the expanded tile is ready, and with it the stage's kpe and scales (the expanding
                // warps waited for the stage before they released the tile).  With two token groups a
                // buffer's previous use may be the other group's tile, not yet filled: a parity wait
                // on xfull alone could then match an older phase.  So wait first until the previous
                // use is released; the use before it (4 tiles back) is this group's own tile or lies
                // in a segment both groups have finished, so that wait is unambiguous, and once the
                // previous use is released xfull is in this use's phase or the one before it.
                const uint32_t xu = tcount / C::kXBufs;
                if (kr == 0) {
                    if (C::kTokenGroups > 1 && xu > 0)
                        ok = wait_phase_flag(&misc->xempty[xb], (xu - 1) & 1, &misc->abort_flag, prm.status, 36);
                    if (ok) ok = wait_phase_flag(&misc->xfull[xb], xu & 1, &misc->abort_flag, prm.status, 34);
                }
                ok = !named_barrier_or(named_bar, 128, !ok || *reinterpret_cast<volatile int*>(&misc->abort_flag));
                if (!ok) break;
                if (kr == 0 && lane == 0) MLA_TRACE_EVENT(2, tcount);
                const uint32_t st_addr = smem_u32(stage_base + sl * C::kStageBytes);
                const uint32_t x_addr = smem_u32(xbase + xb * C::kXBytes);
                const float* scl = reinterpret_cast<const float*>(stage_base + sl * C::kStageBytes + C::kScaleOff);
                // token j of the tile (j < ntok): with 16-token boxes (page size 16) the second box's
                // scales start at float 32
                const int sc_hi = box_rows == kTile ? 0 : 16;
                auto tok_scale = [&](int j) { return scl[j + (j & sc_hi)]; };
                // ---- partial scores over this warp's 144 dims: latent (f16) and rope (bf16) apart
                float sc[4][4], sr[4][4];
#pragma unroll
                for (int n = 0; n < 4; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[n][e] = sr[n][e] = 0.f;
                // k-step ks covers dims kr * 144 + 16 ks: latent (f16, from the expanded tile) for
                // warps 0-2 and the first 5 steps of warp 3, rope (bf16, from the stage) for warp 3's
                // last 4.  Two unrolled loops keep every step's MMA type fixed at compile time.
                auto kstep = [&](int ks, bool rope) {
                    const int kd = kr * 144 + ks * 16;
                    const uint32_t chunk_base = rope ? st_addr + C::kKpeOff : x_addr + (kd >> 6) * C::kXChunkBytes;
                    const int unit0 = (kd & 63) >> 3;
                    uint32_t bf[2][4];
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        const int tk = np * 16 + (lane & 7) + ((lane & 16) ? 8 : 0);
                        ldsm_x4(sw_unit(chunk_base, tk, unit0 + ((lane & 8) ? 1 : 0)), bf[np][0], bf[np][1], bf[np][2],
                                bf[np][3]);
                    }
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        if (np * 16 < ntok) {
                            if (rope) {
                                mma_bf16_16816(sr[2 * np], qa[ks], bf[np][0], bf[np][1]);
                                mma_bf16_16816(sr[2 * np + 1], qa[ks], bf[np][2], bf[np][3]);
                            } else {
                                mma_f16_16816(sc[2 * np], qa[ks], bf[np][0], bf[np][1]);
                                mma_f16_16816(sc[2 * np + 1], qa[ks], bf[np][2], bf[np][3]);
                            }
                        }
                    }
                };
                if (kr < 3) {
#pragma unroll
                    for (int ks = 0; ks < 9; ++ks) kstep(ks, false);
                } else {
#pragma unroll
                    for (int ks = 0; ks < 5; ++ks) kstep(ks, false);
#pragma unroll
                    for (int ks = 5; ks < 9; ++ks) kstep(ks, true);
                }
                // latent part times s_t / sigma_h, plus the rope part -> the group's partial buffer
                {
                    float4* dst = reinterpret_cast<float4*>(part) + kr * 4 * 32;
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        const int j = 8 * n + 2 * c4;
                        const float s0 = j < ntok ? tok_scale(j) : 0.f;
                        const float s1 = j + 1 < ntok ? tok_scale(j + 1) : 0.f;
                        dst[n * 32 + lane] = make_float4(fmaf(sc[n][0], s0 * isg[0], sr[n][0]),
                                                         fmaf(sc[n][1], s1 * isg[0], sr[n][1]),
                                                         fmaf(sc[n][2], s0 * isg[1], sr[n][2]),
                                                         fmaf(sc[n][3], s1 * isg[1], sr[n][3]));
                    }
                }
                if (kr == 0 && lane == 0) MLA_TRACE_EVENT(3, tcount);
                // the tile's largest token scale (every warp of the group the same)
                float tile_c = lane < ntok ? tok_scale(lane) : 0.f;
                tile_c = warp_max(tile_c);
                named_barrier_sync(named_bar, 128);
                float s4[4];
                {
                    const float4* src = reinterpret_cast<const float4*>(part);
                    const float4 a0 = src[(0 * 4 + kr) * 32 + lane], a1 = src[(1 * 4 + kr) * 32 + lane];
                    const float4 a2 = src[(2 * 4 + kr) * 32 + lane], a3 = src[(3 * 4 + kr) * 32 + lane];
                    s4[0] = ((a0.x + a1.x) + a2.x) + a3.x;
                    s4[1] = ((a0.y + a1.y) + a2.y) + a3.y;
                    s4[2] = ((a0.z + a1.z) + a2.z) + a3.z;
                    s4[3] = ((a0.w + a1.w) + a2.w) + a3.w;
                }
                const int tok = kr * 8 + 2 * c4;   // this lane's two tokens
                if (ntok < kTile) {
                    if (tok >= ntok) s4[0] = s4[2] = -INFINITY;
                    if (tok + 1 >= ntok) s4[1] = s4[3] = -INFINITY;
                }
                // ---- running scale maximum: move it (and rescale O) when the tile exceeds it by 16x
                if (tile_c > 16.f * c_run) {
                    const float f = c_run > 0.f ? c_run / tile_c : 0.f;
#pragma unroll
                    for (int n = 0; n < 16; ++n) o[n][0] *= f, o[n][1] *= f, o[n][2] *= f, o[n][3] *= f;
                    c_run = tile_c;
                }
                const float inv_c = c_run > 0.f ? __frcp_rn(c_run) : 0.f;
                const float w0 = tok < ntok ? tok_scale(tok) * inv_c : 0.f;
                const float w1 = tok + 1 < ntok ? tok_scale(tok + 1) * inv_c : 0.f;
                // ---- row maxima, lazy running max, softmax weights (as in the bf16 kernel)
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
                    const uint32_t v0 = pack_f16(p0 * w0, p1 * w1), v1 = pack_f16(p2 * w0, p3 * w1);
                    *reinterpret_cast<uint32_t*>(pbuf + g * C::kPRowBytes + tok * 2) = v0;
                    *reinterpret_cast<uint32_t*>(pbuf + (g + 8) * C::kPRowBytes + tok * 2) = v1;
                }
                named_barrier_sync(named_bar, 128);
                if (kr == 0 && lane == 0) MLA_TRACE_EVENT(4, tcount);
                uint32_t pa[2][4];
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const int prow = (lane & 7) + ((lane & 8) ? 8 : 0);
                    const int pcol = kt * 16 + ((lane & 16) ? 8 : 0);
                    ldsm_x4(smem_u32(pbuf) + prow * C::kPRowBytes + pcol * 2, pa[kt][0], pa[kt][1], pa[kt][2], pa[kt][3]);
                }
                // ---- O[16 x 128 dims of this warp] += P' V (V: the expanded codes; rows past ntok are 0)
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    if (kt * 16 >= ntok) break;
                    const int vt = kt * 16 + (lane & 7) + ((lane & 8) ? 8 : 0);
                    uint32_t vf[8][4];
#pragma unroll
                    for (int dp = 0; dp < 8; ++dp) {
                        const int d0 = kr * 128 + dp * 16;
                        const int un = ((d0 & 63) >> 3) + ((lane & 16) ? 1 : 0);
                        ldsm_x4_t(sw_unit(x_addr + (d0 >> 6) * C::kXChunkBytes, vt, un), vf[dp][0], vf[dp][1], vf[dp][2],
                                  vf[dp][3]);
                    }
#pragma unroll
                    for (int dp = 0; dp < 8; ++dp) {
                        mma_f16_16816(o[2 * dp], pa[kt], vf[dp][0], vf[dp][1]);
                        mma_f16_16816(o[2 * dp + 1], pa[kt], vf[dp][2], vf[dp][3]);
                    }
                }
                __syncwarp();
                if (kr == 0 && lane == 0) MLA_TRACE_EVENT(5, tcount);
                if (lane == 0) {
                    mbar_arrive(&misc->xempty[xb]);
                    mbar_arrive(&misc->empty[sl]);
                }
            }
            if (C::kTokenGroups == 2)
                ok = !named_barrier_or(merge_bar, 256, !ok || *reinterpret_cast<volatile int*>(&misc->abort_flag));
            if (!ok) break;
            const int ctr = (sg.item * prm.head_groups + group_cta) * C::kHeadGroups + hgi;
            int ticket = 0;
            if (sg.slot >= 0 && tg == 0 && gt == 0) ticket = atomicAdd(&prm.counters[ctr], 1);
            // ---- row sums
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
            if (C::kTokenGroups == 2) {
                // ---- merge the token groups: group 1 passes (O, m, l, c) to group 0 through shared
                // memory, group 0 brings both to the larger scale maximum and combines
                float4* xo = reinterpret_cast<float4*>(part_base + (hgi * C::kTokenGroups) * (C::kPartBytes / 4));
                named_barrier_sync(merge_bar, 256);
                if (tg == 1 && kr == 0 && c4 == 0) {
                    misc->tg_m[g] = m_run[0];
                    misc->tg_m[g + 8] = m_run[1];
                    misc->tg_l[g] = l[0];
                    misc->tg_l[g + 8] = l[1];
                    if (g == 0) misc->tg_c = c_run;
                }
                float w0[2] = {1.f, 1.f}, w1[2] = {0.f, 0.f};
                float f0 = 1.f, f1 = 0.f;
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
                            const float c1 = misc->tg_c;
                            const float cm = fmaxf(c_run, c1);
                            f0 = cm > 0.f ? c_run / cm : 0.f;
                            f1 = cm > 0.f ? c1 / cm : 0.f;
                            c_run = cm;
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
                            on[0] = on[0] * (w0[0] * f0) + v.x * (w1[0] * f1);
                            on[1] = on[1] * (w0[0] * f0) + v.y * (w1[0] * f1);
                            on[2] = on[2] * (w0[1] * f0) + v.z * (w1[1] * f1);
                            on[3] = on[3] * (w0[1] * f0) + v.w * (w1[1] * f1);
                        }
                    }
                    named_barrier_sync(merge_bar, 256);
                }
            }
            const bool wide = C::kTokenGroups == 2 && sg.slot >= 0 && si == seg_end - 1;
            if (tg == 1 && !wide) continue;
            if (tg == 0) {
                // ---- epilogue: out = c O / l
                const float inv0 = c_run / l[0], inv1 = c_run / l[1];
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
            }
            if (sg.slot >= 0) {
                // ---- split request: publish, or (last ticket) wait for the others and merge
                const uint32_t mbar = wide ? merge_bar : named_bar;
                const uint32_t nthr = wide ? 256u : 128u;
                if (tg == 0 && gt == 0) misc->merge_flag[hgi] = (ticket == sg.n_slots - 1) ? 1 : 0;
                named_barrier_sync(mbar, nthr);
                if (!misc->merge_flag[hgi]) {
                    if (tg == 0) __threadfence();
                    named_barrier_sync(mbar, nthr);
                    if (tg == 0 && gt == 0) atomicAdd(&prm.ready[ctr], 1);
                } else {
                    if (tg == 0 && gt == 0) {
                        bool done = ld_acquire_gpu(prm.ready + ctr) >= sg.n_slots - 1;
                        const uint64_t tw = global_timer_ns();
                        while (!done && !*reinterpret_cast<volatile int*>(&misc->abort_flag)) {
                            if (global_timer_ns() - tw > kWaitLimitNs) {
                                misc->abort_flag = 1;
                                atomicCAS(prm.status, 0u, kStatusTimeout | 35u);
                                break;
                            }
                            done = ld_acquire_gpu(prm.ready + ctr) >= sg.n_slots - 1;
                        }
                        misc->merge_flag[hgi] = done ? 1 : 2;
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
                    }
                }
                named_barrier_sync(mbar, nthr);
            }
        }
    }
    __syncthreads();
}

}  // namespace mla
