// The decode prologue: the step just before attention in a decode layer (FlashMLA PR #233,
// "What is added": one prologue kernel for RoPE, concat, cache write and quantize-on-write).
//
// For each new token, the query row r = b * qo_len + j: the new tokens are the last qo_len of
// request b's cache, so row r sits at position t = L_b - qo_len + j, in page
// kv_indices[kv_indptr[b] + t / page_size], slot t % page_size.  One CTA per row:
//   * q_pe_out[r, h, :] = rope(q_pe_in[r, h, :], t) for every head h (the rope part of the
//     query; its latent part q_nope is used as it is, so the concat [q_nope | q_pe] is the pair
//     of buffers the decode reads);
//   * kpe_cache[page, slot, :] = rope(kpe_new[r, :], t);
//   * ckv_cache[page, slot, :] = ckv_new[r, :] for a 16-bit cache (bf16, or fp16 with fp16
//     inputs), or for an 8-bit cache, every step in fp32: e4m3, s = absmax / 448 over the
//     token's 512 values and codes = e4m3(x / s) rounded to nearest even with saturation;
//     INT8, s = absmax / 127 and codes = x / s rounded to nearest even, clamped to [-127, 127];
//     ckv_scale[page, slot] = s (s = 0 and zero codes for an all-zero token).
// RoPE ("Benchmarking MLA", FlashInfer issue #700: "partial apply RoPE (only on first
// 64-dimension)") rotates 32 pairs of the 64 rope dims, pair i by the angle of position t with
// frequency i: (x, y) -> (x cos - y sin, x sin + y cos), cos and sin read from the caller's
// table [max_pos, 64] (cos of pairs 0..31, then their sin), so any frequency schedule fits.
// Pair i is dims (2i, 2i + 1) when interleaved, else (i, i + 32).  The rotation runs in fp32
// and rounds to bf16 (fp16 with fp16 inputs).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "mla_decode.h"

namespace {

constexpr int kDimCkv = 512;
constexpr int kDimKpe = 64;
constexpr int kThreads = 128;
constexpr float kE4m3Max = 448.f;
constexpr float kInt8Max = 127.f;

struct PrologueParams {
    const uint16_t* q_pe_in;
    uint16_t* q_pe_out;
    const uint16_t* ckv_new;
    const uint16_t* kpe_new;
    const float* rope;          // [max_pos, 64]
    const int32_t* kv_indices;
    const int32_t* kv_indptr;
    const int32_t* kv_last_page_len;
    uint8_t* ckv_cache;         // bf16 / fp16 values, or e4m3 / INT8 codes
    float* ckv_scale;           // 8-bit caches: [num_pages, page_size]
    uint16_t* kpe_cache;
    int rows, qo_len, h_q, page_size, num_pages, max_pos, kind, interleaved;   // kind: mla_kv_dtype_t
};

// 16-bit values of the inputs: bf16, or IEEE fp16 (f16)
__device__ __forceinline__ float in16_to_f32(uint16_t v, bool f16) {
    return f16 ? __half2float(__ushort_as_half(v)) : __uint_as_float(static_cast<uint32_t>(v) << 16);
}

__device__ __forceinline__ uint16_t f32_to_16(float v, bool f16) {
    return f16 ? __half_as_ushort(__float2half_rn(v)) : __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// rotate pair i of the 64 rope dims at src into dst (both 16-bit), with cos c, sin s
__device__ __forceinline__ void rope_pair(const uint16_t* src, uint16_t* dst, int i, float c, float s,
                                          bool interleaved, bool f16) {
    const int a = interleaved ? 2 * i : i;
    const int b = interleaved ? 2 * i + 1 : i + kDimKpe / 2;
    const float x = in16_to_f32(src[a], f16), y = in16_to_f32(src[b], f16);
    dst[a] = f32_to_16(x * c - y * s, f16);
    dst[b] = f32_to_16(x * s + y * c, f16);
}

__global__ void __launch_bounds__(kThreads) mla_decode_prologue_kernel(PrologueParams p) {
    // The decode that usually follows is launched with programmatic dependent launch: this
    // lets its CTAs start their set-up now; they read the cache only after this grid has
    // completed and its writes are visible (their griddepcontrol.wait).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int b = r / p.qo_len, j = r % p.qo_len;
    const int n = p.kv_indptr[b + 1] - p.kv_indptr[b];
    const int64_t L = n > 0 ? static_cast<int64_t>(n - 1) * p.page_size + p.kv_last_page_len[b] : 0;
    const int64_t t = L - p.qo_len + j;
    if (t < 0 || t >= p.max_pos) return;   // no such position: the row is left untouched
    const float* cs = p.rope + t * kDimKpe;
    const bool il = p.interleaved != 0;
    const bool f16 = p.kind == MLA_KV_F16;
    // the query's rope part, every head
    for (int idx = tid; idx < p.h_q * (kDimKpe / 2); idx += kThreads) {
        const int h = idx / (kDimKpe / 2), i = idx % (kDimKpe / 2);
        const size_t row = (static_cast<size_t>(r) * p.h_q + h) * kDimKpe;
        rope_pair(p.q_pe_in + row, p.q_pe_out + row, i, cs[i], cs[kDimKpe / 2 + i], il, f16);
    }
    const int page = p.kv_indices[p.kv_indptr[b] + static_cast<int>(t / p.page_size)];
    if (page < 0 || page >= p.num_pages) return;   // outside the cache buffers: nothing is written
    const size_t tok = static_cast<size_t>(page) * p.page_size + static_cast<size_t>(t % p.page_size);
    if (tid < kDimKpe / 2)
        rope_pair(p.kpe_new + static_cast<size_t>(r) * kDimKpe, p.kpe_cache + tok * kDimKpe, tid, cs[tid],
                  cs[kDimKpe / 2 + tid], il, f16);
    // the latent: thread tid owns dims [4 tid, 4 tid + 4)
    const uint2 raw = *reinterpret_cast<const uint2*>(p.ckv_new + static_cast<size_t>(r) * kDimCkv + 4 * tid);
    if (p.kind == MLA_KV_BF16 || f16) {
        *reinterpret_cast<uint2*>(p.ckv_cache + (tok * kDimCkv + 4 * tid) * 2) = raw;
        return;
    }
    const bool i8 = p.kind == MLA_KV_INT8;
    const float qmax = i8 ? kInt8Max : kE4m3Max;
    float x[4] = {in16_to_f32(raw.x & 0xffffu, false), in16_to_f32(raw.x >> 16, false),
                  in16_to_f32(raw.y & 0xffffu, false), in16_to_f32(raw.y >> 16, false)};
    float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float wmax[kThreads / 32];
    if ((tid & 31) == 0) wmax[tid >> 5] = m;
    __syncthreads();
    const float absmax = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    const float s = __fdiv_rn(absmax, qmax);
    uint32_t codes = 0;
    if (s > 0.f) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t c;
            if (i8) {   // round half to even, then clamp (|x| <= absmax keeps it within 127 but for rounding)
                const float y = fminf(fmaxf(rintf(__fdiv_rn(x[k], s)), -kInt8Max), kInt8Max);
                c = static_cast<uint32_t>(static_cast<int32_t>(y)) & 0xffu;
            } else {
                const float y = fminf(fmaxf(__fdiv_rn(x[k], s), -kE4m3Max), kE4m3Max);
                c = __nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3) & 0xffu;
            }
            codes |= c << (8 * k);
        }
    }
    *reinterpret_cast<uint32_t*>(p.ckv_cache + tok * kDimCkv + 4 * tid) = codes;
    if (tid == 0) p.ckv_scale[tok] = s;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" mla_status_t mla_decode_prologue(int batch, int qo_len, int h_q, int page_size, mla_kv_dtype_t kv_dtype,
                                            int rope_interleaved, const void* q_pe_in, void* q_pe_out,
                                            const void* ckv_new, const void* kpe_new, const float* rope_cos_sin,
                                            int max_pos, const int32_t* kv_indices, const int32_t* kv_indptr,
                                            const int32_t* kv_last_page_len, void* ckv_cache, float* ckv_scale,
                                            void* kpe_cache, int num_pages, void* cuda_stream) {
    if (batch < 1 || qo_len < 1 || qo_len > 64 || h_q < 1 || h_q > 128 || max_pos < 1 || num_pages < 1)
        return MLA_ERR_INVALID_ARG;
    if (page_size != 16 && page_size != 32 && page_size != 64) return MLA_ERR_UNSUPPORTED;
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3 && kv_dtype != MLA_KV_INT8 && kv_dtype != MLA_KV_F16)
        return MLA_ERR_INVALID_ARG;
    if (!q_pe_in || !q_pe_out || !ckv_new || !kpe_new || !rope_cos_sin || !kv_indices || !kv_indptr ||
        !kv_last_page_len || !ckv_cache || !kpe_cache)
        return MLA_ERR_INVALID_ARG;
    const bool eight = kv_dtype == MLA_KV_FP8_E4M3 || kv_dtype == MLA_KV_INT8;
    if (eight != (ckv_scale != nullptr)) return MLA_ERR_INVALID_ARG;
    if (!aligned(ckv_new, 8) || !aligned(ckv_cache, 8) || !aligned(q_pe_in, 2) || !aligned(q_pe_out, 2) ||
        !aligned(kpe_new, 2) || !aligned(kpe_cache, 2) || !aligned(rope_cos_sin, 4) || (ckv_scale && !aligned(ckv_scale, 4)))
        return MLA_ERR_INVALID_ARG;
    const int64_t rows = static_cast<int64_t>(batch) * qo_len;
    if (rows >= (int64_t(1) << 31) / 128) return MLA_ERR_INVALID_ARG;
    PrologueParams p;
    p.q_pe_in = static_cast<const uint16_t*>(q_pe_in);
    p.q_pe_out = static_cast<uint16_t*>(q_pe_out);
    p.ckv_new = static_cast<const uint16_t*>(ckv_new);
    p.kpe_new = static_cast<const uint16_t*>(kpe_new);
    p.rope = rope_cos_sin;
    p.kv_indices = kv_indices;
    p.kv_indptr = kv_indptr;
    p.kv_last_page_len = kv_last_page_len;
    p.ckv_cache = static_cast<uint8_t*>(ckv_cache);
    p.ckv_scale = ckv_scale;
    p.kpe_cache = static_cast<uint16_t*>(kpe_cache);
    p.rows = static_cast<int>(rows);
    p.qo_len = qo_len;
    p.h_q = h_q;
    p.page_size = page_size;
    p.num_pages = num_pages;
    p.max_pos = max_pos;
    p.kind = static_cast<int>(kv_dtype);
    p.interleaved = rope_interleaved ? 1 : 0;
    mla_decode_prologue_kernel<<<static_cast<unsigned>(rows), kThreads, 0, static_cast<cudaStream_t>(cuda_stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
