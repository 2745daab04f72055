// C ABI of the MLA paged decode library (declared in include/mla_decode.h):
// plan lifetime, workspace commit, tensor-map setup and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "mla_decode.h"
#include "attn.cuh"
#include "attn_e4m3.cuh"
#include "attn_narrow.cuh"
#include "attn_narrow8.cuh"
#include "attn_pair.cuh"
#include "plan.h"

// Tensor maps of the last run's buffers (re-encoded when an address changes).
struct MapCache {
    bool valid = false;
    const void *ckv = nullptr, *kpe = nullptr, *qn = nullptr, *qp = nullptr, *scale = nullptr;
    int num_pages = 0;
    CUtensorMap m_ckv, m_kpe, m_qp, m_v, m_scale;
};

struct mla_plan_s {
    mla::PlanData d;
    MapCache maps;
    uint64_t* trace = nullptr;    // device timeline buffer (builds with MLA_TRACE only)
    std::vector<uint8_t> image;   // header bytes copied to the workspace by commit
    void* pinned = nullptr;       // pinned staging copy of `image`
    std::vector<void*> committed; // workspaces this plan has been committed to
    int test_withhold = 0;        // test builds (MLA_TEST_HOOKS) only
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, box [box_rows, 64 columns],
// 128-byte swizzle (one box row = 128 bytes).
bool make_map_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of the ckv cache for the narrow kernel: dims (64 dims, rows, 8 chunks) with
// strides (2 B, 1024 B, 128 B); a box (64, box_rows, 8) copies box_rows whole rows into
// shared memory as [chunk][row][128 B] with the 128-byte swizzle.
bool make_map_ckv_chunked(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, 8};
    cuuint64_t strides[2] = {mla::kDimCkv * 2, 128};
    cuuint32_t box[3] = {64, box_rows, 8};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Key view of the ckv cache for the 128-head kernel: dims (64 dims, 8 rows, 8 chunks, rows / 8
// row groups) with strides (2 B, 1024 B, 128 B, 8192 B); a box (64, 8, 4, page / 8) copies one
// page's rows of 4 chunks (256 dims) as [row group][chunk][8 rows][128 B] with the 128-byte
// swizzle, so consecutive pages' boxes make one K-major operand of 4 chunks whose 8-row groups
// lie 4 KB apart.  The values read the same view: chunks 4 * half.. as the MN-major operand,
// 64-dim groups 1 KB apart and 8-token groups 4 KB apart.
bool make_map_ckv_rg4(CUtensorMap* map, const void* base, uint64_t rows, uint32_t page) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {64, 8, 8, rows / 8};
    cuuint64_t strides[3] = {mla::kDimCkv * 2, 128, 8 * mla::kDimCkv * 2};
    cuuint32_t box[4] = {64, 8, 4, page / 8};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 codes of the ckv cache ([rows, 512] bytes) for the e4m3 kernel: a 2-D view with boxes
// of 128 code columns (one 128-dim chunk) x box_rows rows, 128-byte swizzle.
bool make_map_codes(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint32_t es[2] = {1, 1};
    cuuint64_t dims[2] = {mla::kDimCkv, rows};
    cuuint64_t strides[1] = {mla::kDimCkv};
    cuuint32_t box[2] = {128, box_rows};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 1-D fp32 view of the per-token scales of an e4m3 cache ([num_pages * page_size]), box of one
// page; coordinates past either end read zeros.
bool make_map_scale(CUtensorMap* map, const float* base, uint64_t n, uint32_t box) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[1] = {n};
    cuuint64_t strides[1] = {n * 4};   // unused for a 1-D map
    cuuint32_t bx[1] = {box};
    cuuint32_t es[1] = {1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, const_cast<float*>(base), dims, strides, bx, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void build_image(mla_plan_s* p) {
    const auto& L = p->d.layout;
    p->image.assign(L.header_bytes, 0);
    std::memcpy(p->image.data() + L.off_unit_ptr, p->d.unit_ptr.data(), sizeof(int32_t) * p->d.unit_ptr.size());
    if (!p->d.segments.empty())
        std::memcpy(p->image.data() + L.off_segments, p->d.segments.data(),
                    sizeof(mla::Segment) * p->d.segments.size());
}

// Launch with programmatic stream serialization: the kernel's prologue (barriers, TMEM, its
// slice of the plan) may overlap the tail of the previous kernel in the stream; the kernels
// wait for that kernel (griddepcontrol.wait) before they touch any buffer of the caller.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int threads, int smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int HG, bool F16>
cudaError_t launch_narrow(const mla_plan_s* p, const CUtensorMap& ckv, const CUtensorMap& kpe, const mla::AttnParams& prm,
                          const void* q_nope, const void* q_pe, cudaStream_t stream) {
    using C = mla::NarrowCfg<HG>;
    cudaError_t e = cudaFuncSetAttribute(mla::mla_decode_narrow_kernel<HG, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = p->d.num_units * p->d.head_groups;
    return launch_pdl(mla::mla_decode_narrow_kernel<HG, F16>, grid, C::kThreads, C::kSmemBytes, stream, ckv, kpe, prm,
                      static_cast<const uint16_t*>(q_nope), static_cast<const uint16_t*>(q_pe));
}

template <int HG>
cudaError_t launch_narrow8(const mla_plan_s* p, const MapCache& mc, const mla::AttnParams& prm, const void* q_nope,
                           const void* q_pe, cudaStream_t stream) {
    using C = mla::Narrow8Cfg<HG>;
    cudaError_t e = cudaFuncSetAttribute(mla::mla_decode_narrow8_kernel<HG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = p->d.num_units * p->d.head_groups;
    return launch_pdl(mla::mla_decode_narrow8_kernel<HG>, grid, C::kThreads, C::kSmemBytes, stream, mc.m_ckv, mc.m_kpe,
                      mc.m_scale, prm, static_cast<const uint16_t*>(q_nope), static_cast<const uint16_t*>(q_pe));
}

cudaError_t launch_e4m3(const mla_plan_s* p, const MapCache& mc, const mla::AttnParams& prm, const void* q_nope,
                        const void* q_pe, cudaStream_t stream) {
    using C = mla::E4m3Cfg;
    cudaError_t e = cudaFuncSetAttribute(mla::mla_decode_e4m3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = p->d.num_units * p->d.head_groups;
    return launch_pdl(mla::mla_decode_e4m3_kernel, grid, C::kThreads, C::kSmemBytes, stream, mc.m_ckv, mc.m_kpe,
                      mc.m_scale, prm, static_cast<const uint16_t*>(q_nope), static_cast<const uint16_t*>(q_pe));
}

template <int HQ, bool F16>
cudaError_t launch_pair(const mla_plan_s* p, const MapCache& mc, const mla::AttnParams& prm, const void* q_nope,
                        cudaStream_t stream) {
    using C = mla::PairCfg;
    cudaError_t e = cudaFuncSetAttribute(mla::mla_decode_pair_kernel<HQ, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = 2 * p->d.num_units;   // clusters of two CTAs (the kernel's cluster dimensions)
    return launch_pdl(mla::mla_decode_pair_kernel<HQ, F16>, grid, C::kThreads, C::kSmemBytes, stream, mc.m_ckv, mc.m_kpe,
                      mc.m_qp, mc.m_v, prm, static_cast<const uint16_t*>(q_nope));
}

// Argument checks, tensor maps and the launch shared by mla_decode_run and
// mla_decode_run_noalloc; `ws` is the committed workspace (device).
mla_status_t run_checked(mla_plan_t plan, const void* q_nope, const void* q_pe, const void* ckv_cache,
                         const float* ckv_scale, const void* kpe_cache, int num_pages, const int32_t* kv_indices,
                         const int32_t* kv_indptr, float sm_scale, void* out, float* lse, uint8_t* ws,
                         cudaStream_t stream, uint64_t* trace) {
    const auto& d = plan->d;
    const bool f8 = d.kv_dtype == MLA_KV_FP8_E4M3 || d.kv_dtype == MLA_KV_INT8;   // 8-bit codes
    const auto& L = d.layout;
    // tensor maps depend only on the buffer addresses: re-encode when they change
    MapCache& mc = plan->maps;
    if (!mc.valid || mc.ckv != ckv_cache || mc.kpe != kpe_cache || mc.qn != q_nope || mc.qp != q_pe ||
        mc.scale != ckv_scale || mc.num_pages != num_pages) {
        const uint64_t rows = static_cast<uint64_t>(num_pages) * d.page_size;
        const uint64_t qrows = static_cast<uint64_t>(d.rows) * d.h_q;
        const uint32_t hg = static_cast<uint32_t>(d.heads_per_cta);
        // box rows: a whole page for the tcgen05 kernel, a 32-token ring stage at most for the narrow one
        const uint32_t box = (d.narrow || d.narrow8) ? std::min(d.page_size, mla::kNarrowStageTok) : d.page_size;
        // the narrow kernel takes a whole 32-token stage of ckv in one 3-D box when a page holds it
        const bool chunked = d.narrow && box == static_cast<uint32_t>(mla::kNarrowStageTok);
        bool ok_ckv;
        if (f8)
            ok_ckv = make_map_codes(&mc.m_ckv, ckv_cache, rows, box);
        else if (d.pair)
            ok_ckv = make_map_ckv_rg4(&mc.m_ckv, ckv_cache, rows, static_cast<uint32_t>(d.page_size));
        else
            ok_ckv = chunked ? make_map_ckv_chunked(&mc.m_ckv, ckv_cache, rows, box)
                             : make_map_bf16(&mc.m_ckv, ckv_cache, mla::kDimCkv, rows, box);
        mc.valid = ok_ckv && make_map_bf16(&mc.m_kpe, kpe_cache, mla::kDimKpe, rows, box) &&
                   make_map_bf16(&mc.m_qp, q_pe, mla::kDimKpe, qrows, d.pair ? 128 : hg) &&
                   (!d.pair || make_map_ckv_rg4(&mc.m_v, ckv_cache, rows, static_cast<uint32_t>(d.page_size))) &&
                   (!f8 || make_map_scale(&mc.m_scale, ckv_scale, rows, box));
        if (!mc.valid) return MLA_ERR_CUDA;
        mc.ckv = ckv_cache;
        mc.kpe = kpe_cache;
        mc.qn = q_nope;
        mc.qp = q_pe;
        mc.scale = ckv_scale;
        mc.num_pages = num_pages;
    }
    mla::AttnParams prm;
    prm.unit_ptr = reinterpret_cast<const int32_t*>(ws + L.off_unit_ptr);
    prm.segments = reinterpret_cast<const mla::Segment*>(ws + L.off_segments);
    prm.kv_indices = kv_indices;
    prm.kv_indptr = kv_indptr;
    prm.ckv = static_cast<const uint8_t*>(ckv_cache);
    prm.kpe = static_cast<const uint8_t*>(kpe_cache);
    prm.out = static_cast<float*>(out);
    prm.lse = lse;
    prm.part_o = reinterpret_cast<float*>(ws + L.off_part_o);
    prm.part_lse = reinterpret_cast<float*>(ws + L.off_part_lse);
    prm.ckv_scale = ckv_scale;
    prm.counters = reinterpret_cast<int32_t*>(ws + L.off_counters);
    prm.ready = prm.counters + static_cast<size_t>(d.num_split) * (d.h_q / 16);
    prm.status = reinterpret_cast<uint32_t*>(ws + L.off_status);
    prm.trace = trace;
    prm.scale_log2 = sm_scale * 1.4426950408889634f;
    prm.h_q = d.h_q;
    prm.page_size = d.page_size;
    prm.head_groups = d.head_groups;
    prm.num_pages = num_pages;
    prm.out_bf16 = d.out_dtype == MLA_OUT_BF16 ? 1 : 0;
    prm.test_withhold = plan->test_withhold;
    cudaError_t e;
    if (d.narrow8) {
        e = d.heads_per_cta == 16 ? launch_narrow8<16>(plan, mc, prm, q_nope, q_pe, stream)
                                  : launch_narrow8<32>(plan, mc, prm, q_nope, q_pe, stream);
    } else if (d.e4m3) {
        e = launch_e4m3(plan, mc, prm, q_nope, q_pe, stream);
    } else if (d.narrow) {
        if (d.f16)
            e = d.h_q == 16 ? launch_narrow<16, true>(plan, mc.m_ckv, mc.m_kpe, prm, q_nope, q_pe, stream)
                            : launch_narrow<32, true>(plan, mc.m_ckv, mc.m_kpe, prm, q_nope, q_pe, stream);
        else
            e = d.h_q == 16 ? launch_narrow<16, false>(plan, mc.m_ckv, mc.m_kpe, prm, q_nope, q_pe, stream)
                            : launch_narrow<32, false>(plan, mc.m_ckv, mc.m_kpe, prm, q_nope, q_pe, stream);
    } else if (d.pair) {
        if (d.f16)
            e = d.h_q == 128 ? launch_pair<128, true>(plan, mc, prm, q_nope, stream)
                             : launch_pair<64, true>(plan, mc, prm, q_nope, stream);
        else
            e = d.h_q == 128 ? launch_pair<128, false>(plan, mc, prm, q_nope, stream)
                             : launch_pair<64, false>(plan, mc, prm, q_nope, stream);
    } else {
        return MLA_ERR_UNSUPPORTED;   // the plan admits no other head count
    }
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// Host-side argument checks common to both run entry points.
mla_status_t check_run_args(mla_plan_t plan, const void* q_nope, const void* q_pe, const void* ckv_cache,
                            const float* ckv_scale, const void* kpe_cache, int num_pages, const int32_t* kv_indices,
                            const int32_t* kv_indptr, const int32_t* kv_last_page_len, float sm_scale,
                            const void* out, const float* lse) {
    if (!plan || !q_nope || !q_pe || !ckv_cache || !kpe_cache || !kv_indices || !kv_indptr || !kv_last_page_len ||
        !out || !lse || num_pages < 1)
        return MLA_ERR_INVALID_ARG;
    const auto& d = plan->d;
    if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(ckv_cache) || !aligned16(kpe_cache) ||
        !aligned16(out) || !aligned16(lse))
        return MLA_ERR_INVALID_ARG;
    if (!std::isfinite(sm_scale)) return MLA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_pages) * d.page_size >= (int64_t(1) << 31)) return MLA_ERR_INVALID_ARG;
    const bool eight = d.kv_dtype == MLA_KV_FP8_E4M3 || d.kv_dtype == MLA_KV_INT8;
    if (!eight && ckv_scale != nullptr) return MLA_ERR_INVALID_ARG;
    if (eight && (ckv_scale == nullptr || !aligned16(ckv_scale))) return MLA_ERR_INVALID_ARG;
    return MLA_OK;
}

void* noalloc_scratch_address();   // the fixed array of mla_decode_run_noalloc (end of this file)

}  // namespace

extern "C" {

mla_status_t mla_decode_plan(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host, int batch,
                             int h_q, int page_size, int num_sms, mla_kv_dtype_t kv_dtype, mla_plan_t* plan_out) {
    return mla_decode_plan_ex(kv_indptr_host, kv_last_page_len_host, batch, 1, 0, h_q, page_size, num_sms, kv_dtype,
                              MLA_OUT_F32, plan_out);
}

mla_status_t mla_decode_plan_ex(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host, int batch,
                                int qo_len, int causal, int h_q, int page_size, int num_sms,
                                mla_kv_dtype_t kv_dtype, mla_out_dtype_t out_dtype, mla_plan_t* plan_out) {
    if (!plan_out) return MLA_ERR_INVALID_ARG;
    mla::PlanData d;
    const int rc = mla::build_plan(kv_indptr_host, kv_last_page_len_host, batch, qo_len, causal != 0, h_q, page_size,
                                   num_sms, static_cast<int>(kv_dtype), static_cast<int>(out_dtype), &d);
    if (rc == 1) return MLA_ERR_INVALID_ARG;
    if (rc == 2) return MLA_ERR_UNSUPPORTED;
    auto* p = new (std::nothrow) mla_plan_s;
    if (!p) return MLA_ERR_INVALID_ARG;
    p->d = std::move(d);
    build_image(p);
    *plan_out = p;
    return MLA_OK;
}

size_t mla_decode_plan_workspace_bytes(mla_plan_t plan) { return plan ? plan->d.layout.total_bytes : 0; }

mla_status_t mla_decode_plan_commit(mla_plan_t plan, void* workspace_dev, size_t workspace_bytes,
                                    void* cuda_stream) {
    if (!plan || !workspace_dev) return MLA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0) return MLA_ERR_INVALID_ARG;
    if (workspace_bytes < plan->d.layout.total_bytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (!plan->pinned) {
        if (cudaMallocHost(&plan->pinned, plan->image.size()) != cudaSuccess) {
            plan->pinned = nullptr;
            return MLA_ERR_CUDA;
        }
        std::memcpy(plan->pinned, plan->image.data(), plan->image.size());
    }
    if (cudaMemcpyAsync(workspace_dev, plan->pinned, plan->image.size(), cudaMemcpyHostToDevice,
                        static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (std::find(plan->committed.begin(), plan->committed.end(), workspace_dev) == plan->committed.end())
        plan->committed.push_back(workspace_dev);
    return MLA_OK;
}

mla_status_t mla_decode_run(mla_plan_t plan, const void* q_nope, const void* q_pe, const void* ckv_cache,
                            const float* ckv_scale, const void* kpe_cache, int num_pages,
                            const int32_t* kv_indices, const int32_t* kv_indptr,
                            const int32_t* kv_last_page_len, float sm_scale, void* out, float* lse,
                            void* workspace_dev, void* cuda_stream) {
    mla_status_t st = check_run_args(plan, q_nope, q_pe, ckv_cache, ckv_scale, kpe_cache, num_pages, kv_indices,
                                     kv_indptr, kv_last_page_len, sm_scale, out, lse);
    if (st != MLA_OK) return st;
    if (!workspace_dev) return MLA_ERR_INVALID_ARG;
    if (std::find(plan->committed.begin(), plan->committed.end(), workspace_dev) == plan->committed.end())
        return MLA_ERR_NOT_COMMITTED;
    if (plan->d.segments.empty()) return MLA_OK;
    return run_checked(plan, q_nope, q_pe, ckv_cache, ckv_scale, kpe_cache, num_pages, kv_indices, kv_indptr,
                       sm_scale, out, lse, static_cast<uint8_t*>(workspace_dev),
                       static_cast<cudaStream_t>(cuda_stream), plan->trace);
}

#ifdef MLA_TRACE
// Debug builds only: device buffer of 4 * 8 * 256 uint64 timestamps filled by the next runs.
void mla_debug_set_trace(mla_plan_t plan, void* dev_buf) {
    if (plan) plan->trace = static_cast<uint64_t*>(dev_buf);
}
#endif

#ifdef MLA_TEST_HOOKS
// Test builds only: with withhold != 0 the bf16 narrow-head kernel's CTA 0 never fills its first
// ring stage, so a consumer's bounded wait runs out (a failure made without any fault).
void mla_debug_set_withhold(mla_plan_t plan, int withhold) {
    if (plan) plan->test_withhold = withhold;
}
#endif

int mla_plan_num_launches(mla_plan_t plan) { return (plan && !plan->d.segments.empty()) ? 1 : 0; }

mla_status_t mla_decode_device_status(mla_plan_t plan, void* workspace_dev, void* cuda_stream) {
    if (!plan) return MLA_ERR_INVALID_ARG;
    // NULL: the status word of the fixed array mla_decode_run_noalloc works in
    if (!workspace_dev) workspace_dev = noalloc_scratch_address();
    if (!workspace_dev) return MLA_ERR_CUDA;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, static_cast<uint8_t*>(workspace_dev) + plan->d.layout.off_status, sizeof word,
                        cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
    if (word == 0) return MLA_OK;
    if (cudaMemsetAsync(static_cast<uint8_t*>(workspace_dev) + plan->d.layout.off_status, 0, sizeof word, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return MLA_ERR_CUDA;
    return MLA_ERR_DEVICE_TIMEOUT;
}

int mla_plan_num_ctas(mla_plan_t plan) {
    return plan ? plan->d.num_units * plan->d.head_groups * (plan->d.pair ? 2 : 1) : 0;
}
int mla_plan_num_units(mla_plan_t plan) { return plan ? plan->d.num_units : 0; }
int mla_plan_num_segments(mla_plan_t plan) { return plan ? static_cast<int>(plan->d.segments.size()) : 0; }
int mla_plan_num_partials(mla_plan_t plan) { return plan ? plan->d.num_partials : 0; }
int mla_plan_heads_per_cta(mla_plan_t plan) { return plan ? plan->d.heads_per_cta : 0; }
int mla_plan_segment_cost_tiles(mla_plan_t plan) { return plan ? plan->d.segment_cost : 0; }
int mla_plan_num_rows(mla_plan_t plan) { return plan ? plan->d.rows : 0; }

int mla_plan_get_segments(mla_plan_t plan, int32_t* segments, int32_t* unit_ptr) {
    if (!plan) return 0;
    const auto& d = plan->d;
    if (segments)
        for (size_t i = 0; i < d.segments.size(); ++i) {
            segments[4 * i + 0] = d.segments[i].b;
            segments[4 * i + 1] = d.segments[i].t_begin;
            segments[4 * i + 2] = d.segments[i].t_end;
            segments[4 * i + 3] = d.segments[i].slot;
        }
    if (unit_ptr) std::copy(d.unit_ptr.begin(), d.unit_ptr.end(), unit_ptr);
    return static_cast<int>(d.segments.size());
}

void mla_plan_destroy(mla_plan_t plan) {
    if (!plan) return;
    if (plan->pinned) cudaFreeHost(plan->pinned);
    delete plan;
}

const char* mla_status_string(mla_status_t status) {
    switch (status) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported h_q, page_size or cache type";
        case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MLA_ERR_CUDA: return "CUDA error";
        case MLA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case MLA_ERR_NOT_COMMITTED: return "plan not committed to this workspace";
        default: return "unknown status";
    }
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// Decode without any device allocation by the caller or the library.
//
// The workspace (work-list header, split partials, status word) lives in a fixed, file-scope
// device array instead of caller-allocated memory.  It exists once per GPU that loads this
// library and stays allocated until the process exits.  Host code may not use its address
// directly (in host code `g_noalloc_scratch` names a host-side stand-in), so the device address
// is fetched with cudaGetSymbolAddress once per device, with that device current, and cached.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on first use).  The address
// is kept for the life of the process: after a cudaDeviceReset it is stale, and the calls that use
// it (mla_decode_run_noalloc, mla_decode_device_status with no workspace) must not be made again.
void* noalloc_scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" size_t mla_decode_noalloc_max_workspace_bytes(void) { return kNoAllocScratchBytes; }

extern "C" mla_status_t mla_decode_run_noalloc(mla_plan_t plan, const void* q_nope, const void* q_pe,
                                               const void* ckv_cache, const float* ckv_scale, const void* kpe_cache,
                                               int num_pages, const int32_t* kv_indices, const int32_t* kv_indptr,
                                               const int32_t* kv_last_page_len, float sm_scale, void* out,
                                               float* lse, void* cuda_stream) {
    mla_status_t st = check_run_args(plan, q_nope, q_pe, ckv_cache, ckv_scale, kpe_cache, num_pages, kv_indices,
                                     kv_indptr, kv_last_page_len, sm_scale, out, lse);
    if (st != MLA_OK) return st;
    if (plan->d.layout.total_bytes > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* ws = static_cast<uint8_t*>(noalloc_scratch_address());
    if (!ws) return MLA_ERR_CUDA;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    // The plan's header (work list, zeroed status word and merge counters) is copied in on every
    // call, straight from the plan's host image: the array keeps the previous call's contents.
    if (cudaMemcpyAsync(ws, plan->image.data(), plan->image.size(), cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (plan->d.segments.empty()) return MLA_OK;
    return run_checked(plan, q_nope, q_pe, ckv_cache, ckv_scale, kpe_cache, num_pages, kv_indices, kv_indptr,
                       sm_scale, out, lse, ws, stream, nullptr);
}
