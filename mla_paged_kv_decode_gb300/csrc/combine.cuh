// Deterministic merge of split-KV partials (FlashMLA PR #233: "balanced
// scheduler, deterministic combine").  For a request split into k pieces with
// partial results (o_i, lse_i), in the fixed slot order i = 0..k-1:
//
//   M = max_i lse_i,  w_i = exp(lse_i - M),
//   out = sum_i w_i o_i / sum_i w_i,   lse = M + ln sum_i w_i.
//
// One CTA of 128 threads per (request item, head); each thread owns four
// consecutive latent dims (one float4).  A request with no tokens gets out = 0
// and lse = -inf.  Partials are small (h_q * 2 KB per piece) and were written
// just before by the attention kernel, so they are normally L2 resident.
#pragma once

#include <cstdint>

#include "plan.h"

namespace mla {

__global__ void __launch_bounds__(128) mla_decode_combine_kernel(const CombineItem* __restrict__ items,
                                                                  const float* __restrict__ part_o,
                                                                  const float* __restrict__ part_lse,
                                                                  float* __restrict__ out, float* __restrict__ lse,
                                                                  int h_q) {
    const CombineItem it = items[blockIdx.x];
    const int h = blockIdx.y;
    const int d4 = threadIdx.x;  // float4 index, 0..127
    float4* o4 = reinterpret_cast<float4*>(out + (static_cast<size_t>(it.b) * h_q + h) * kDimCkv) + d4;
    if (it.n_slots == 0) {
        *o4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (d4 == 0) lse[static_cast<size_t>(it.b) * h_q + h] = -INFINITY;
        return;
    }
    float M = -INFINITY;
    for (int i = 0; i < it.n_slots; ++i)
        M = fmaxf(M, part_lse[static_cast<size_t>(it.slot_begin + i) * h_q + h]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    for (int i = 0; i < it.n_slots; ++i) {
        const size_t s = static_cast<size_t>(it.slot_begin + i) * h_q + h;
        const float w = expf(part_lse[s] - M);
        const float4 v = reinterpret_cast<const float4*>(part_o + s * kDimCkv)[d4];
        wsum += w;
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    const float inv = 1.f / wsum;
    *o4 = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (d4 == 0) lse[static_cast<size_t>(it.b) * h_q + h] = M + logf(wsum);
}

}  // namespace mla
