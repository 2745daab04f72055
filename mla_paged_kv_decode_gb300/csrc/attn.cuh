// Pieces shared by the decode kernels (attn_narrow.cuh: 16/32 heads, attn_pair.cuh: 64/128
// heads): the kernel parameters, bounded mbarrier waits, the debug timeline, the tile cursor
// over a CTA's segments and the split-KV merge.
//
// Absorbed MLA decode is MQA with one KV head: key [ckv | kpe] (576), value ckv (512)
// ("Benchmarking MLA", FlashInfer issue #700).  The plan cuts each request's tokens into
// segments; a segment that is one piece of a split request writes its normalised partial
// (o, lse) into the workspace, and the CTA whose arrival on the request's counter is the last
// merges all pieces in slot order (FlashMLA PR #233, "deterministic combine"):
//   M = max_i lse_i, w_i = exp(lse_i - M), out = sum_i w_i o_i / sum_i w_i,
//   lse = M + ln sum_i w_i,
// then resets the counter for the next run.  The arithmetic does not depend on which CTA
// merges, so results are bit-identical from run to run.
//
// Every mbarrier wait is bounded; on expiry a kernel records a status code, drains its
// in-flight copies and MMAs, frees TMEM and returns.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "plan.h"
#include "ptx.cuh"

namespace mla {

constexpr uint32_t kStatusTimeout = 0x100u;       // OR-ed with the wait site id
// Time without progress before a wait gives up: 4 s (a test build may set a shorter limit).
#ifndef MLA_WAIT_LIMIT_NS
#define MLA_WAIT_LIMIT_NS 4000000000ull
#endif
constexpr uint64_t kWaitLimitNs = MLA_WAIT_LIMIT_NS;

struct AttnParams {
    const int32_t* unit_ptr;      // [num_units + 1]
    const Segment* segments;      // [num_segments]
    const int32_t* kv_indices;
    const int32_t* kv_indptr;
    const uint8_t* ckv;           // cache base addresses (L2 prefetch of whole pages)
    const uint8_t* kpe;
    float* out;                   // [rows, h_q, 512]: fp32, or bf16 at the same address when out_bf16
    float* lse;                   // [rows, h_q] fp32
    float* part_o;                // [num_partials, h_q, 512]
    float* part_lse;              // [num_partials, h_q]
    const float* ckv_scale;       // e4m3 cache: fp32 scale per token [num_pages * page_size], else null
    int32_t* counters;            // arrivals per (split request, 16- or 32-head block)
    int32_t* ready;               // narrow kernel: pieces of each counter whose partial is written
    uint32_t* status;
    uint64_t* trace;              // per-tile event timestamps when built with MLA_TRACE, else unused
    float scale_log2;             // sm_scale * log2(e)
    int h_q;
    int page_size;
    int head_groups;
    int num_pages;                // pages in the cache buffers
    int out_bf16;                 // the final output is bf16 (partials stay fp32)
    int test_withhold;            // test builds (MLA_TEST_HOOKS) only: CTA 0 withholds its first stage
};

// A destination of fp32 results: a buffer base and its element type.  The final output may
// be bf16 (rounded to nearest even); partials are always fp32.  Element offsets are counted
// from the base in elements of the buffer's own type.
struct OutDst {
    float* base;
    bool bf16;
};

__device__ __forceinline__ OutDst final_out(const AttnParams& prm) { return OutDst{prm.out, prm.out_bf16 != 0}; }
__device__ __forceinline__ OutDst fp32_dst(float* base) { return OutDst{base, false}; }

__device__ __forceinline__ void st_out(OutDst d, size_t i, float v) {
    if (d.bf16)
        reinterpret_cast<__nv_bfloat16*>(d.base)[i] = __float2bfloat16_rn(v);
    else
        d.base[i] = v;
}

__device__ __forceinline__ void st_out2(OutDst d, size_t i, float a, float b) {   // i even
    if (d.bf16)
        *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(d.base) + i) = __floats2bfloat162_rn(a, b);
    else
        *reinterpret_cast<float2*>(d.base + i) = make_float2(a, b);
}

__device__ __forceinline__ void st_out4(OutDst d, size_t i, float4 v) {   // i a multiple of 4
    if (d.bf16) {
        __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(d.base) + i);
        p[0] = __floats2bfloat162_rn(v.x, v.y);
        p[1] = __floats2bfloat162_rn(v.z, v.w);
    } else {
        *reinterpret_cast<float4*>(d.base + i) = v;
    }
}

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

// Optional pipeline timeline (compiled in with -DMLA_TRACE): CTAs 0..3 record the
// global timer at event `ev` of their tile `idx` into prm.trace[cta][ev][idx].  With
// -DMLA_TRACE_CLOCK the stamps are the SM's cycle counter instead (finer, but comparable only
// between stamps taken on one SM).
#ifdef MLA_TRACE
#ifdef MLA_TRACE_CLOCK
#define MLA_TRACE_NOW() static_cast<uint64_t>(clock64())
#else
#define MLA_TRACE_NOW() global_timer_ns()
#endif
// the two CTAs whose per-tile events are recorded: MLA_TRACE_FIRST and the next one
#ifndef MLA_TRACE_FIRST
#define MLA_TRACE_FIRST 0
#endif
#define MLA_TRACE_EVENT(ev, idx)                                                              \
    do {                                                                                      \
        if (prm.trace && blockIdx.x >= MLA_TRACE_FIRST && blockIdx.x < MLA_TRACE_FIRST + 2 && \
            (idx) < 256)                                                                      \
            prm.trace[((blockIdx.x - MLA_TRACE_FIRST) * 8 + (ev)) * 256 + (idx)] =            \
                MLA_TRACE_NOW();                                                              \
    } while (0)
// CTA 0 only: a timestamp per unit of work (a ring slot fill, ...) in the area of CTAs 2 and 3,
// lane `ln` (0..3) of 1024 entries each.
#define MLA_TRACE_UNIT(ln, idx)                                                               \
    do {                                                                                      \
        if (prm.trace && blockIdx.x == 0 && (idx) < 1024)                                     \
            prm.trace[2 * 8 * 256 + (ln) * 1024 + (idx)] = MLA_TRACE_NOW();                   \
    } while (0)
// CTA 1 only: the same per-unit stamps, in 4 lanes of 1024 entries after the milestones.
#define MLA_TRACE_UNIT1(ln, idx)                                                              \
    do {                                                                                      \
        if (prm.trace && blockIdx.x == 1 && (idx) < 1024)                                     \
            prm.trace[4 * 8 * 256 + gridDim.x * 8 + (ln) * 1024 + (idx)] = MLA_TRACE_NOW();   \
    } while (0)
// Every CTA also records 8 milestones (entry, producer done, ...) after the per-tile area.
#define MLA_TRACE_CTA(k)                                                                      \
    do {                                                                                      \
        if (prm.trace) prm.trace[4 * 8 * 256 + blockIdx.x * 8 + (k)] = MLA_TRACE_NOW();       \
    } while (0)
// A second set of 8 milestones per CTA (after CTA 1's unit lanes); the stamp is read after
// `dep` is available, so it marks the arrival of the loads `dep` depends on.
#define MLA_TRACE_CTA2(k, dep)                                                                \
    do {                                                                                      \
        if (prm.trace) {                                                                      \
            uint64_t t_;                                                                      \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_) : "f"(dep));                 \
            prm.trace[4 * 8 * 256 + gridDim.x * 8 + 4 * 1024 + blockIdx.x * 8 + (k)] = t_;    \
        }                                                                                     \
    } while (0)
#else
#define MLA_TRACE_EVENT(ev, idx) \
    do {                         \
    } while (0)
#define MLA_TRACE_CTA(k) \
    do {                 \
    } while (0)
#define MLA_TRACE_CTA2(k, dep) \
    do {                       \
    } while (0)
#define MLA_TRACE_UNIT(ln, idx) \
    do {                        \
    } while (0)
#define MLA_TRACE_UNIT1(ln, idx) \
    do {                         \
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
// give identical bits.  The loads are issued in batches (several pieces and heads at once)
// so the merge costs a few memory round trips rather than one per (piece, head).
// NTHR threads (tid 0..NTHR-1) call it together and synchronise on named barrier `bar`.
// Scratch in shared memory: s_max[NH], s_inv[NH], s_w[max(8 * NH, 128)].
//
// This general form serves any number of pieces.  Its outputs go by chunks of 8 pieces
// (their weights staged in shared memory) and, beyond 16 heads or with 256 threads, by blocks
// of 8 heads, each chunk's loads in rounds of 4 pieces x 8 heads (2 pieces for 16 heads, whose
// two 8-head blocks run side by side on 256 threads); 128 threads and 16 heads load one piece
// of all 16 heads a round.
// Every output sums the same products in the same order (pieces in slot order, from 0) with
// 128 or 256 threads, so the two forms give identical bits.  The up-to-8 form below takes
// fewer rounds.
template <int NH, int NTHR>
__device__ __forceinline__ void merge_split_pieces_chunked(const AttnParams& prm, int b, int slot_begin, int n_slots,
                                                           int head0, int tid, uint32_t bar, float* s_max,
                                                           float* s_inv, float* s_w) {
    static_assert(NH % 16 == 0 && (NTHR == 128 || (NTHR == 256 && NH == 16)), "merge layout");
    constexpr int kTph = 128 / NH;     // threads per head in the lse pass (threads 0..127)
    constexpr int kBlocks = NTHR / 128;   // 8-head blocks merged side by side
    // pieces per round of loads: 4 for the many heads of the two-CTA kernel (its threads hold 255
    // registers), 2 for 16 heads on 256 threads (within the warp-MMA kernels' registers)
    constexpr int kHB = 8, kPB = NH > 16 ? 4 : 2, kChunk = 8;
    const size_t hq = static_cast<size_t>(prm.h_q);
    if (tid < 128) {
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
    const OutDst od = final_out(prm);
    const int t = tid & 127, g = tid >> 7;
    const size_t o0 = (static_cast<size_t>(b) * hq + head0) * kDimCkv + 4 * t;
    if constexpr (NH == 16 && NTHR == 128) {
        // ---- outputs, 128 threads and 16 heads: thread t owns dims [4 t, 4 t + 4) of every head,
        // one piece (all 16 heads) per round of loads, within the warp-MMA kernels' registers
        float4 acc[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int c0 = 0; c0 < n_slots; c0 += kChunk) {
            {
                const int i = tid / 16, h = tid % 16;   // weight of piece c0 + i for head h
                float w = 0.f;
                if (c0 + i < n_slots)
                    w = expf(__ldcg(prm.part_lse + (slot_begin + c0 + i) * hq + head0 + h) - s_max[h]) * s_inv[h];
                s_w[tid] = w;
            }
            named_barrier_sync(bar, NTHR);
            const int n = min(kChunk, n_slots - c0);
#pragma unroll 1
            for (int i = 0; i < n; ++i) {
                const float4* src = reinterpret_cast<const float4*>(prm.part_o + ((slot_begin + c0 + i) * hq + head0) *
                                                                                    kDimCkv) + t;
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
        for (int h = 0; h < 16; ++h) st_out4(od, o0 + static_cast<size_t>(h) * kDimCkv, acc[h]);
    } else {
    // ---- outputs: thread t owns dims [4 t, 4 t + 4) of its block's 8 heads
#pragma unroll 1
    for (int hb0 = 0; hb0 < NH; hb0 += kHB * kBlocks) {
        const int hb = hb0 + g * kHB;   // this thread's first head
        float4 acc[kHB];
#pragma unroll
        for (int h = 0; h < kHB; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int c0 = 0; c0 < n_slots; c0 += kChunk) {
            if (tid < kBlocks * kChunk * kHB) {   // weight of piece c0 + i for head hb0 + 8 gb + h
                const int gb = tid / (kChunk * kHB), i = (tid / kHB) % kChunk, h = tid % kHB;
                const int head = hb0 + gb * kHB + h;
                float w = 0.f;
                if (c0 + i < n_slots)
                    w = expf(__ldcg(prm.part_lse + (slot_begin + c0 + i) * hq + head0 + head) - s_max[head]) *
                        s_inv[head];
                s_w[tid] = w;
            }
            named_barrier_sync(bar, NTHR);
            const int cn = min(kChunk, n_slots - c0);
#pragma unroll 1
            for (int p0 = 0; p0 < cn; p0 += kPB) {
                float4 v[kPB][kHB];
#pragma unroll
                for (int i = 0; i < kPB; ++i)
#pragma unroll
                    for (int h = 0; h < kHB; ++h)
                        v[i][h] = (p0 + i < cn)
                                      ? __ldcg(reinterpret_cast<const float4*>(
                                                   prm.part_o + ((slot_begin + c0 + p0 + i) * hq + head0 + hb + h) *
                                                                    kDimCkv) + t)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < kPB; ++i) {
                    if (p0 + i >= cn) break;
#pragma unroll
                    for (int h = 0; h < kHB; ++h) {
                        const float w = s_w[(g * kChunk + p0 + i) * kHB + h];
                        acc[h].x = fmaf(w, v[i][h].x, acc[h].x);
                        acc[h].y = fmaf(w, v[i][h].y, acc[h].y);
                        acc[h].z = fmaf(w, v[i][h].z, acc[h].z);
                        acc[h].w = fmaf(w, v[i][h].w, acc[h].w);
                    }
                }
            }
            named_barrier_sync(bar, NTHR);   // s_w is rewritten next
        }
#pragma unroll
        for (int h = 0; h < kHB; ++h) st_out4(od, o0 + static_cast<size_t>(hb + h) * kDimCkv, acc[h]);
    }
    }
}

// The same merge for up to 8 pieces: every thread loads the lse of its pieces once and
// computes their weights itself, and the outputs go by blocks of 8 heads x 4 pieces whose
// loads are all in flight together.  The first block's loads are issued before the lse
// reduction.  Same sums, same fixed orders (pieces in slot order) as the general form.
template <int NH, int NTHR>
__device__ __forceinline__ void merge_split_pieces(const AttnParams& prm, int b, int slot_begin, int n_slots,
                                                   int head0, int tid, uint32_t bar, float* s_max, float* s_inv,
                                                   float* s_w) {
    static_assert(NTHR == 128 && NH % 16 == 0 && NTHR % NH == 0, "merge layout");
    constexpr int kMax = 8;            // pieces served here
    constexpr int kTph = NTHR / NH;    // threads per head in the lse pass
    constexpr int kPer = kMax / kTph;  // pieces per thread in the lse pass
    constexpr int kHB = 8, kPB = 4;    // output block: heads x pieces with their loads in flight together
    if (n_slots > kMax) {
        merge_split_pieces_chunked<NH, NTHR>(prm, b, slot_begin, n_slots, head0, tid, bar, s_max, s_inv, s_w);
        return;
    }
    const size_t hq = static_cast<size_t>(prm.h_q);
    auto piece_o = [&](int i, int h) {   // this thread's 4 dims of head h, piece i
        return reinterpret_cast<const float4*>(prm.part_o + ((slot_begin + i) * hq + head0 + h) * kDimCkv) + tid;
    };
    float4 v[kPB][kHB];
    auto load_block = [&](int hb, int p0) {
#pragma unroll
        for (int i = 0; i < kPB; ++i)
#pragma unroll
            for (int h = 0; h < kHB; ++h)
                v[i][h] = (p0 + i < n_slots) ? __ldcg(piece_o(p0 + i, hb + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    load_block(0, 0);   // in flight during the lse pass
    {
        const int h = tid / kTph, sub = tid % kTph;
        float x[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = sub + kTph * j;
            x[j] = i < n_slots ? __ldcg(prm.part_lse + (slot_begin + i) * hq + head0 + h) : -INFINITY;
        }
        float m = x[0];
#pragma unroll
        for (int j = 1; j < kPer; ++j) m = fmaxf(m, x[j]);
#pragma unroll
        for (int o = kTph / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        // every piece has a finite lse (a non-empty token range), so m is finite
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < kPer; ++j) sum += (sub + kTph * j < n_slots) ? expf(x[j] - m) : 0.f;
#pragma unroll
        for (int o = kTph / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = 1.f / sum;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = sub + kTph * j;
            if (i < n_slots) s_w[i * NH + h] = expf(x[j] - m) * inv;
        }
        if (sub == 0) {
            s_max[h] = m;
            s_inv[h] = inv;
            prm.lse[static_cast<size_t>(b) * hq + head0 + h] = m + logf(sum);
        }
    }
    named_barrier_sync(bar, NTHR);
    const OutDst od = final_out(prm);
    const size_t o0 = (static_cast<size_t>(b) * hq + head0) * kDimCkv + 4 * tid;
#pragma unroll 1
    for (int hb = 0; hb < NH; hb += kHB) {
        float4 acc[kHB];
#pragma unroll
        for (int h = 0; h < kHB; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int p0 = 0; p0 < n_slots; p0 += kPB) {
            if (hb != 0 || p0 != 0) load_block(hb, p0);
#pragma unroll
            for (int i = 0; i < kPB; ++i) {
                if (p0 + i >= n_slots) break;
#pragma unroll
                for (int h = 0; h < kHB; ++h) {
                    const float w = s_w[(p0 + i) * NH + hb + h];
                    acc[h].x = fmaf(w, v[i][h].x, acc[h].x);
                    acc[h].y = fmaf(w, v[i][h].y, acc[h].y);
                    acc[h].z = fmaf(w, v[i][h].z, acc[h].z);
                    acc[h].w = fmaf(w, v[i][h].w, acc[h].w);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < kHB; ++h) st_out4(od, o0 + static_cast<size_t>(hb + h) * kDimCkv, acc[h]);
    }
}

// The merge of up to 8 pieces of 16 heads by 256 threads: threads [128 k, 128 k + 128) take
// heads [8 k, 8 k + 8), so the loads of every piece (up to 4) of both head blocks go out in one
// round, together with the lse loads.  Threads 0..127 run the lse pass of
// merge_split_pieces<16, 128>, and every output sums the same products in the same order as
// there: the two forms give identical bits.  More than 8 pieces: threads 0..127 run the
// general form on the 128-thread barrier `bar128`, the others return.
__device__ __forceinline__ void merge_split_pieces_wide16(const AttnParams& prm, int b, int slot_begin, int n_slots,
                                                          int head0, int tid, uint32_t bar256, uint32_t bar128,
                                                          float* s_max, float* s_inv, float* s_w) {
    constexpr int NH = 16, kMax = 8, kTph = 8, kHB = 8, kPB = 4;
    if (n_slots > kMax) {
        merge_split_pieces_chunked<NH, 256>(prm, b, slot_begin, n_slots, head0, tid, bar256, s_max, s_inv, s_w);
        return;
    }
    const size_t hq = static_cast<size_t>(prm.h_q);
    const int t = tid & 127, hb = (tid >> 7) * kHB;
    auto piece_o = [&](int i, int h) {   // this thread's 4 dims of head h, piece i
        return reinterpret_cast<const float4*>(prm.part_o + ((slot_begin + i) * hq + head0 + h) * kDimCkv) + t;
    };
    float4 v[kPB][kHB];
    auto load_block = [&](int p0) {
#pragma unroll
        for (int i = 0; i < kPB; ++i)
#pragma unroll
            for (int h = 0; h < kHB; ++h)
                v[i][h] = (p0 + i < n_slots) ? __ldcg(piece_o(p0 + i, hb + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    if (tid == 0) MLA_TRACE_CTA2(0, 0.f);
    load_block(0);   // in flight during the lse pass
    if (tid < 128) {
        const int h = tid / kTph, sub = tid % kTph;
        const float x = sub < n_slots ? __ldcg(prm.part_lse + (slot_begin + sub) * hq + head0 + h) : -INFINITY;
        float m = x;
#pragma unroll
        for (int o = kTph / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = sub < n_slots ? expf(x - m) : 0.f;
#pragma unroll
        for (int o = kTph / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = 1.f / sum;
        if (sub < n_slots) s_w[sub * NH + h] = expf(x - m) * inv;
        if (sub == 0) {
            s_max[h] = m;
            s_inv[h] = inv;
            prm.lse[static_cast<size_t>(b) * hq + head0 + h] = m + logf(sum);
        }
    }
    named_barrier_sync(bar256, 256);
    if (tid == 0) MLA_TRACE_CTA2(1, s_w[0]);
    float4 acc[kHB];
#pragma unroll
    for (int h = 0; h < kHB; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int p0 = 0; p0 < n_slots; p0 += kPB) {
        if (p0 != 0) load_block(p0);
#pragma unroll
        for (int i = 0; i < kPB; ++i) {
            if (p0 + i >= n_slots) break;
#pragma unroll
            for (int h = 0; h < kHB; ++h) {
                const float w = s_w[(p0 + i) * NH + hb + h];
                acc[h].x = fmaf(w, v[i][h].x, acc[h].x);
                acc[h].y = fmaf(w, v[i][h].y, acc[h].y);
                acc[h].z = fmaf(w, v[i][h].z, acc[h].z);
                acc[h].w = fmaf(w, v[i][h].w, acc[h].w);
            }
        }
    }
    if (tid == 0) MLA_TRACE_CTA2(2, acc[0].x);
    const OutDst od = final_out(prm);
    const size_t o0 = (static_cast<size_t>(b) * hq + head0) * kDimCkv + 4 * t;
#pragma unroll
    for (int h = 0; h < kHB; ++h) st_out4(od, o0 + static_cast<size_t>(hb + h) * kDimCkv, acc[h]);
    if (tid == 0) MLA_TRACE_CTA2(3, 0.f);
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

}  // namespace mla
