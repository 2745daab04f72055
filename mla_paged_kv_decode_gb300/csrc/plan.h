// Host-side split-KV plan: work list layout shared by the scheduler (plan.cpp),
// the C ABI (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

namespace mla {

constexpr int kTileTokens = 128;   // tokens per attention tile (UMMA M of the score MMA)
constexpr int kDimCkv = 512;
constexpr int kDimKpe = 64;

// One (request, token range) piece of work.  slot < 0: the piece is the whole
// request and the kernel writes out/lse directly; otherwise it writes the
// partial (out, lse) to partial slot `slot`.
struct Segment {
    int32_t b, t_begin, t_end, slot;
};

// One request the combine kernel finalises: merges partial slots
// [slot_begin, slot_begin + n_slots), or zero-fills when n_slots == 0.
struct CombineItem {
    int32_t b, slot_begin, n_slots, pad;
};

struct PlanLayout {
    size_t off_status = 0;      // uint32 status word
    size_t off_unit_ptr = 0;    // int32 [num_units + 1]
    size_t off_segments = 0;    // Segment [num_segments]
    size_t off_items = 0;       // CombineItem [num_items]
    size_t header_bytes = 0;    // bytes copied by commit
    size_t off_part_lse = 0;    // fp32 [num_partials, h_q]
    size_t off_part_o = 0;      // fp32 [num_partials, h_q, 512]
    size_t total_bytes = 0;
};

struct PlanData {
    int batch = 0, h_q = 0, page_size = 0, num_sms = 0, kv_dtype = 0;
    int heads_per_cta = 0, head_groups = 0, num_units = 0;
    std::vector<int32_t> unit_ptr;
    std::vector<Segment> segments;
    std::vector<CombineItem> items;
    int num_partials = 0;
    PlanLayout layout;
};

// Returns 0 on success, 1 invalid argument, 2 unsupported.
int build_plan(const int32_t* kv_indptr, const int32_t* kv_last_page_len, int batch, int h_q, int page_size,
               int num_sms, int kv_dtype, PlanData* out);

// Heads handled by one CTA for a given h_q (0 if unsupported).
int heads_per_cta_for(int h_q, int kv_dtype);

}  // namespace mla
