/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA paged-KV decode library.
 *
 * The operation is absorbed-weight Multi-head Latent Attention decode: multi-
 * query attention with one shared KV head whose key is [ckv (512) | kpe (64)]
 * and whose value is ckv itself ("Benchmarking MLA", FlashInfer issue #700:
 * "what we actually need is a fused-rope MQA kernel"; for the matrix-absorbed
 * kernel qk_head_dim = 512 + 64 and v_head_dim = 512).  For request b, head h:
 *
 *     x_t = sm_scale * (q_nope[b,h,:] . ckv_t + q_pe[b,h,:] . kpe_t)
 *     out[b,h,:] = sum_t softmax(x)_t * ckv_t,   lse[b,h] = ln sum_t exp(x_t)
 *
 * over the request's cached tokens t.  The cache is paged as in "perf: MLA
 * decode kernel implemented by CuTe targeted to SM80" (FlashInfer PR #844):
 * ckv [num_pages, page_size, 512], kpe [num_pages, page_size, 64]; request b
 * owns pages kv_indices[kv_indptr[b] .. kv_indptr[b+1]) in logical order, and
 * its last page holds kv_last_page_len[b] tokens.  Token t is in page
 * kv_indices[kv_indptr[b] + t / page_size], slot t % page_size.
 *
 * The split-KV scheduling (a host "plan" that balances work over the SMs)
 * and the deterministic merge of split partials follow FlashMLA PR #233
 * ("balanced scheduler, deterministic combine, graph-safe API"); the 8-bit
 * cache follows the same page ("FP8 e4m3 ... with one scale per token (644
 * instead of 1152 bytes per token), dequantized inside the kernel").
 *
 * Conventions for every call below
 *   - Device pointers are CUDA device addresses on the current device; host
 *     pointers are ordinary host memory.  The library never frees or keeps
 *     caller memory beyond the call, except that a plan keeps its own host
 *     copy of the work list (and a pinned staging buffer) until
 *     mla_plan_destroy.
 *   - All tensors are dense, row-major, contiguous.
 *   - bf16 means IEEE bfloat16 bit patterns (uint16); fp32 is IEEE float.
 *   - Errors are returned as mla_status_t; nothing is thrown across the ABI,
 *     no call aborts the process.
 *   - cuda_stream is a cudaStream_t passed as void* (NULL = legacy default).
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mla_plan_s* mla_plan_t; /* opaque, host-owned */

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,         /* malformed sizes, indptr not monotone, last_page_len out of range */
    MLA_ERR_UNSUPPORTED = 2,         /* h_q or page_size outside the supported set */
    MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace smaller than mla_decode_plan_workspace_bytes */
    MLA_ERR_CUDA = 4,                /* a CUDA runtime/driver call or a launch failed */
    MLA_ERR_DEVICE_TIMEOUT = 5,      /* a kernel's bounded wait ran out (read by mla_decode_device_status) */
    MLA_ERR_NOT_COMMITTED = 6        /* mla_decode_run before mla_decode_plan_commit */
} mla_status_t;

typedef enum {
    MLA_KV_BF16 = 0,      /* ckv bf16 [num_pages, page_size, 512] */
    MLA_KV_FP8_E4M3 = 1,  /* ckv uint8 e4m3 codes [num_pages, page_size, 512] + fp32 scale [num_pages, page_size] */
    MLA_KV_INT8 = 2,      /* ckv int8 codes (two's complement) [num_pages, page_size, 512] + fp32 scale
                             [num_pages, page_size]; token t's latent is scale[t] * code[t, :] */
    MLA_KV_F16 = 3        /* fp16 inputs: ckv fp16 [num_pages, page_size, 512], and q_nope, q_pe and kpe
                             are IEEE fp16 too (instead of bf16) */
} mla_kv_dtype_t;

typedef enum {
    MLA_OUT_F32 = 0,   /* out fp32 [rows, h_q, 512] */
    MLA_OUT_BF16 = 1   /* out bf16 [rows, h_q, 512], each value the fp32 result rounded to nearest even */
} mla_out_dtype_t;

/* Build a balanced split-KV work list (host only, no device call).
 *
 * Work is measured in tokens.  Requests are laid out in order, cut into
 * tiles of the kernel's size (32 tokens for a bf16 cache with h_q 16 or 32,
 * else 128), and the tile sequence is partitioned into contiguous
 * ranges of near-equal cost, one per CTA slot; a request cut across slots
 * becomes several split pieces whose partial (out, lse) are merged after
 * the attention kernel (FlashMLA PR #233, "balanced scheduler").
 *
 *   kv_indptr_host        host int32 [batch + 1], kv_indptr_host[0] == 0, non-decreasing
 *   kv_last_page_len_host host int32 [batch]; in [1, page_size] for a request with pages,
 *                         ignored (may be anything) for a request with no pages
 *   batch                 >= 1
 *   h_q                   query heads per request: 16, 32, 64 or 128
 *   page_size             16, 32 or 64
 *   num_sms               streaming multiprocessors to plan for (> 0), e.g. 152 on GB300
 *   kv_dtype              cache element type the plan will be run with
 *   plan_out              receives the new plan; untouched on error
 * Returns MLA_OK, MLA_ERR_INVALID_ARG or MLA_ERR_UNSUPPORTED.
 * The plan depends only on these host arrays, so it may be reused across
 * layers and replays while they are unchanged; the contents of kv_indices
 * (physical page placement) may change freely between runs. */
mla_status_t mla_decode_plan(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host, int batch,
                             int h_q, int page_size, int num_sms, mla_kv_dtype_t kv_dtype, mla_plan_t* plan_out);

/* mla_decode_plan with several query tokens per request and a choice of output type.
 *
 * A request may decode qo_len new tokens at once (the pages' tests carry
 * batch_size * qo_len query rows, "perf: MLA decode kernel implemented by CuTe
 * targeted to SM80").  The new tokens are the last qo_len tokens of the
 * request's cache.  Query token j (0-based) of request b is query row
 * r = b * qo_len + j of q_nope / q_pe / out / lse, which then hold
 * rows = batch * qo_len rows:
 *   q_nope [rows, h_q, 512], q_pe [rows, h_q, 64], out [rows, h_q, 512], lse [rows, h_q].
 * Row r attends to request b's first L_b tokens, or with causal != 0 to its
 * first max(0, L_b - (qo_len - 1 - j)) tokens: each new token sees the cache
 * up to and including itself.  A row with no tokens gets out = 0, lse = -inf.
 * Each row streams its request's pages itself: the cache is read qo_len times.
 *
 *   qo_len     1 .. 64
 *   causal     0 or 1 (no effect when qo_len == 1)
 *   out_dtype  MLA_OUT_F32, or MLA_OUT_BF16: out holds bf16 values, each the fp32
 *              result rounded to nearest even; lse stays fp32
 * The other arguments and the return codes are those of mla_decode_plan, which
 * equals this call with qo_len 1, causal 0 and MLA_OUT_F32. */
mla_status_t mla_decode_plan_ex(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host, int batch,
                                int qo_len, int causal, int h_q, int page_size, int num_sms,
                                mla_kv_dtype_t kv_dtype, mla_out_dtype_t out_dtype, mla_plan_t* plan_out);

/* Device workspace the plan needs (bytes, a multiple of 256): the work list,
 * the split partials and a status word.  0 for a NULL plan. */
size_t mla_decode_plan_workspace_bytes(mla_plan_t plan);

/* Copy the plan's work list into the caller's device workspace with one
 * cudaMemcpyAsync on cuda_stream, and clear its status word.  workspace_dev must
 * be 256-byte aligned and at least mla_decode_plan_workspace_bytes(plan) long;
 * it is owned by the caller and must stay alive and untouched by others while
 * runs of this plan are in flight.  Commit once per (plan, workspace) pair,
 * before mla_decode_run.  Returns MLA_OK, MLA_ERR_INVALID_ARG,
 * MLA_ERR_WORKSPACE_TOO_SMALL or MLA_ERR_CUDA. */
mla_status_t mla_decode_plan_commit(mla_plan_t plan, void* workspace_dev, size_t workspace_bytes,
                                    void* cuda_stream);

/* Enqueue one decode on cuda_stream: a single kernel launch.  Each CTA runs
 * its slot of the plan; a split request's pieces write partial (out, lse) to
 * the workspace and the CTA that finishes the request's last piece merges
 * them in slot order (FlashMLA PR #233, "deterministic combine"), so the
 * result does not depend on which CTA merges.
 *
 *   q_nope           device bf16 [batch, h_q, 512] ([rows, h_q, 512] for a plan with qo_len > 1)
 *   q_pe             device bf16 [batch, h_q, 64]  ([rows, h_q, 64])
 *   ckv_cache        device bf16 [num_pages, page_size, 512], or uint8 e4m3 codes of the
 *                    same shape for MLA_KV_FP8_E4M3
 *   ckv_scale        NULL for bf16; device fp32 [num_pages, page_size] for e4m3
 *                    (token t's ckv is ckv_scale[t] * e4m3(code))
 *   kpe_cache        device bf16 [num_pages, page_size, 64]
 *   num_pages        pages in the cache buffers (bounds the tensor maps; a page index
 *                    outside [0, num_pages) reads zeros instead of memory)
 *   kv_indices       device int32 [kv_indptr[batch]]
 *   kv_indptr        device int32 [batch + 1], same values the plan was built from
 *   kv_last_page_len device int32 [batch],     same values the plan was built from
 *   sm_scale         softmax scale applied to q.k (e.g. 1/sqrt(192))
 *   out              device fp32 [batch, h_q, 512], or bf16 when the plan was made with
 *                    MLA_OUT_BF16 ([rows, h_q, 512] for a plan with qo_len > 1)
 *   lse              device fp32 [batch, h_q] ([rows, h_q]), natural log of sum_t exp(x_t);
 *                    -inf and out = 0 for a request with no tokens
 *   workspace_dev    the workspace passed to mla_decode_plan_commit
 * Every device buffer needs 16-byte alignment.  Slots past kv_last_page_len
 * and pages no request references are never used (they may hold NaN).
 * The call allocates nothing, never synchronises and reads no device data on
 * the host, so it may be captured in a CUDA graph; results are bit-identical
 * for the same plan and inputs.  Returns MLA_OK, MLA_ERR_INVALID_ARG,
 * MLA_ERR_NOT_COMMITTED or MLA_ERR_CUDA (launch failure). */
mla_status_t mla_decode_run(mla_plan_t plan, const void* q_nope, const void* q_pe, const void* ckv_cache,
                            const float* ckv_scale, const void* kpe_cache, int num_pages,
                            const int32_t* kv_indices, const int32_t* kv_indptr,
                            const int32_t* kv_last_page_len, float sm_scale, void* out, float* lse,
                            void* workspace_dev, void* cuda_stream);

/* Kernel launches mla_decode_run issues for this plan (1, or 0 when no request has work). */
int mla_plan_num_launches(mla_plan_t plan);

/* Synchronise cuda_stream and read the workspace's status word: MLA_OK, or
 * MLA_ERR_DEVICE_TIMEOUT when a kernel gave up on a bounded wait (its outputs
 * are then undefined).  The word is cleared after reading.  workspace_dev NULL
 * reads the status word of the fixed array mla_decode_run_noalloc uses on the
 * current device; read it after that call and before the next one, which resets
 * it.  Returns MLA_OK, MLA_ERR_DEVICE_TIMEOUT, MLA_ERR_INVALID_ARG (NULL plan)
 * or MLA_ERR_CUDA. */
mla_status_t mla_decode_device_status(mla_plan_t plan, void* workspace_dev, void* cuda_stream);

/* Introspection (host only, for tests and tools). */
int mla_plan_num_ctas(mla_plan_t plan);       /* attention CTAs launched per run */
int mla_plan_num_units(mla_plan_t plan);      /* work units (CTA slots, or CTA pairs for 128 heads) */
int mla_plan_num_segments(mla_plan_t plan);   /* (request, token range) pieces */
int mla_plan_num_partials(mla_plan_t plan);   /* split pieces that go through the combine */
int mla_plan_heads_per_cta(mla_plan_t plan);
/* Partition cost, in tiles (32 tokens for a bf16 cache with h_q <= 32, else 128), that the balanced plan
 * charges for each request start after the first: CTA slots are cut so that tiles plus
 * these costs are equal to within one tile. */
int mla_plan_segment_cost_tiles(mla_plan_t plan);
/* Query rows of out / lse: batch * qo_len. */
int mla_plan_num_rows(mla_plan_t plan);
/* Copy the work list: for segment i, out[4i..4i+3] = (query row, token_begin, token_end,
 * partial slot or -1), the query row being the request with qo_len 1; unit_ptr[u] ..
 * unit_ptr[u+1] are unit u's segments.  Either pointer may be NULL.  Returns the number
 * of segments. */
int mla_plan_get_segments(mla_plan_t plan, int32_t* segments, int32_t* unit_ptr);

/* Decode for callers that cannot allocate device memory: cudaMalloc may be off
 * limits (an allocator that must not be re-entered, a memory pool fixed at start-up,
 * or a framework that owns every device allocation).  This call takes no workspace;
 * it allocates nothing and calls no cudaMalloc, cudaFree or other allocating routine.
 * The pages describe no counterpart to this call: it is an alternative to mla_decode_plan_commit +
 * mla_decode_run with the same arguments and results (minus workspace_dev).
 *
 * The workspace is a fixed device array inside this library, of
 * mla_decode_noalloc_max_workspace_bytes() bytes (16 MiB), present on every GPU that
 * loads the library until the process exits.  A plan whose
 * mla_decode_plan_workspace_bytes exceeds it is rejected with
 * MLA_ERR_WORKSPACE_TOO_SMALL.  Each call first copies the plan's work list (and
 * zeroed merge counters and status word) into the array on cuda_stream, straight from
 * the plan's own pageable host memory, then launches the decode.  The first call on a
 * device also looks up the array's device address (cudaGetSymbolAddress) and keeps it
 * for the life of the process; make no call after a cudaDeviceReset, which leaves the
 * kept address stale.
 * All calls share the one array: calls whose work may overlap on the GPU (different
 * streams, or different host threads) race and corrupt each other's partials; order
 * them on one stream.  A bounded wait that ran out is reported by
 * mla_decode_device_status(plan, NULL, stream), read before the next call.
 * Returns the codes of mla_decode_run, or MLA_ERR_WORKSPACE_TOO_SMALL. */
mla_status_t mla_decode_run_noalloc(mla_plan_t plan, const void* q_nope, const void* q_pe, const void* ckv_cache,
                                    const float* ckv_scale, const void* kpe_cache, int num_pages,
                                    const int32_t* kv_indices, const int32_t* kv_indptr,
                                    const int32_t* kv_last_page_len, float sm_scale, void* out, float* lse,
                                    void* cuda_stream);
/* Size of the fixed workspace array mla_decode_run_noalloc uses (bytes). */
size_t mla_decode_noalloc_max_workspace_bytes(void);

/* The decode prologue: one launch that prepares the new tokens before the decode
 * (FlashMLA PR #233: "one prologue kernel (RoPE, concat, cache write,
 * quantize-on-write)").  The new tokens are the last qo_len tokens of each request,
 * so kv_indptr / kv_last_page_len already count them (the same arrays the plan is
 * built from); row r = b * qo_len + j is token j of request b, at position
 * t = L_b - qo_len + j in page kv_indices[kv_indptr[b] + t / page_size], slot
 * t % page_size.  For each row:
 *   q_pe_out[r, h, :]      = rope(q_pe_in[r, h, :], t) for every head h
 *   kpe_cache[page, slot]  = rope(kpe_new[r, :], t)
 *   ckv_cache[page, slot]  = ckv_new[r, :]               (MLA_KV_BF16, MLA_KV_F16)
 *   or, MLA_KV_FP8_E4M3 (quantise on write, every step in fp32):
 *     s = max_i |ckv_new[r, i]| / 448, ckv_scale[page, slot] = s,
 *     ckv_cache[page, slot, i] = e4m3(clamp(ckv_new[r, i] / s, -448, 448)), rounded to
 *     nearest even (s = 0 and codes 0 when the token is all zeros);
 *   or, MLA_KV_INT8: s = max_i |ckv_new[r, i]| / 127, ckv_scale[page, slot] = s,
 *     ckv_cache[page, slot, i] = clamp(ckv_new[r, i] / s, -127, 127) rounded to nearest even
 *     (s = 0 and codes 0 when the token is all zeros).
 * With MLA_KV_F16 every 16-bit buffer here (q_pe_in/out, ckv_new, kpe_new, the caches) holds
 * IEEE fp16 values and the rotation rounds to fp16; otherwise they are bf16.
 * q_nope needs no work: the decode reads [q_nope | q_pe] as two buffers.
 * rope(x, t) rotates 32 pairs of the 64 rope dims ("partial apply RoPE (only on first
 * 64-dimension)", "Benchmarking MLA", FlashInfer issue #700): pair i, (x, y) ->
 * (x c - y s, x s + y c) with c = rope_cos_sin[t * 64 + i], s = rope_cos_sin[t * 64 + 32 + i],
 * computed in fp32 and rounded to bf16.  Pair i is dims (2i, 2i + 1) when
 * rope_interleaved != 0, else (i, i + 32).
 *
 *   batch, qo_len      requests (>= 1) and new tokens per request (1 .. 64)
 *   h_q, page_size     1 .. 128 heads; 16, 32 or 64
 *   kv_dtype           the cache type (ckv_scale NULL for bf16 / fp16, required for e4m3 / INT8)
 *   q_pe_in, q_pe_out  device bf16 [batch * qo_len, h_q, 64]; may be the same buffer
 *   ckv_new, kpe_new   device bf16 [batch * qo_len, 512] (8-byte aligned), [batch * qo_len, 64]
 *   rope_cos_sin       device fp32 [max_pos, 64]
 *   kv_indices, kv_indptr, kv_last_page_len   device int32, as for mla_decode_run
 *   ckv_cache, ckv_scale, kpe_cache           device caches, written in place
 *   num_pages          pages in the cache buffers
 * A row whose position is negative (a request shorter than qo_len) or >= max_pos is left
 * untouched; a page index outside [0, num_pages) is not written.  One kernel launch on
 * cuda_stream, no allocation, no synchronisation.  Returns MLA_OK, MLA_ERR_INVALID_ARG,
 * MLA_ERR_UNSUPPORTED or MLA_ERR_CUDA. */
mla_status_t mla_decode_prologue(int batch, int qo_len, int h_q, int page_size, mla_kv_dtype_t kv_dtype,
                                 int rope_interleaved, const void* q_pe_in, void* q_pe_out, const void* ckv_new,
                                 const void* kpe_new, const float* rope_cos_sin, int max_pos,
                                 const int32_t* kv_indices, const int32_t* kv_indptr,
                                 const int32_t* kv_last_page_len, void* ckv_cache, float* ckv_scale,
                                 void* kpe_cache, int num_pages, void* cuda_stream);

void mla_plan_destroy(mla_plan_t plan);

/* Static string for a status code. */
const char* mla_status_string(mla_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
