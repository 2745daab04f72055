// Host-side split-KV plan: work list layout shared by the scheduler (plan.cpp),
// the C ABI (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

namespace mla {

constexpr int kTileTokens = 128;   // tokens per tile of the tcgen05 kernels (64/128 heads, e4m3 cache)
constexpr int kNarrowTileTokens = 32;  // tokens per tile of the narrow-head (warp MMA) kernel
// Partition cost of a unit's every segment after its first, in tiles: what a CTA that moves
// on to another request pays for the further segment's prologue and epilogue, measured on
// GB300 against the time of one tile.
#ifndef MLA_NARROW_SEGMENT_COST
#define MLA_NARROW_SEGMENT_COST 4
#endif
constexpr int kNarrowSegmentCost = MLA_NARROW_SEGMENT_COST;
constexpr int kSegmentCost = 1;
// The last piece's merge of a split request, in quarter tiles per piece: about a tile's time for
// the warp-MMA kernels (32-token tiles) and the two-CTA kernel (a 128-head piece is 256 KB), a
// quarter tile for the e4m3 kernel (128-token tiles, 16-head pieces of 32 KB).
constexpr int kMergeCostQuarterTiles = 4;
constexpr int kMergeCostQuarterTilesE4m3 = 1;
constexpr int kDimCkv = 512;
constexpr int kDimKpe = 64;

// One (query row, token range) piece of work.  `b` is the query row (q, out and lse are
// indexed by it: row b * qo_len + j is query token j of request b) and `kv` the request
// whose pages are read; with one query token per request they are equal.  slot < 0: the
// piece is the whole row and the kernel writes out/lse directly (t_begin == t_end == 0 for
// a row with no tokens: out = 0, lse = -inf); otherwise it writes the partial (out, lse)
// to partial slot `slot`, and the CTA that finishes the row's last piece merges slots
// [slot_begin, slot_begin + n_slots) using the arrival counter `item`.
struct Segment {
    int32_t b, t_begin, t_end, slot;
    int32_t item, slot_begin, n_slots, kv;
};

struct PlanLayout {
    size_t off_status = 0;      // uint32 status word
    size_t off_unit_ptr = 0;    // int32 [num_units + 1]
    size_t off_segments = 0;    // Segment [num_segments]
    size_t off_counters = 0;    // int32 [2][num_split_requests * h_q / 16]: arrival tickets, then
                                //   pieces whose partial is written (narrow kernel); zero between runs
    size_t header_bytes = 0;    // bytes copied by commit
    size_t off_part_lse = 0;    // fp32 [num_partials, h_q]
    size_t off_part_o = 0;      // fp32 [num_partials, h_q, 512]
    size_t total_bytes = 0;
};

struct PlanData {
    int batch = 0, h_q = 0, page_size = 0, num_sms = 0, kv_dtype = 0;
    int qo_len = 1;                   // query tokens per request
    bool causal = false;              // query token j of qo_len sees the first L - (qo_len - 1 - j) tokens
    int out_dtype = 0;                // 0: fp32 out, 1: bf16 out
    int rows = 0;                     // query rows: batch * qo_len
    int heads_per_cta = 0, head_groups = 0, num_units = 0;
    int tile_tokens = 0;              // plan granularity = the kernel's tile
    bool narrow = false;              // bf16 cache, h_q <= 32: warp-MMA kernel
    bool pair = false;                // h_q 64/128, bf16 cache: two-CTA cluster kernel, 2 CTAs per unit
    bool e4m3 = false;                // e4m3 cache: tcgen05 kind::f8f6f4 kernel, 16 heads per CTA
    bool narrow8 = false;             // INT8 cache: codes expanded to f16 in the CTA, warp-MMA kernel,
                                      //   16 or 32 heads per CTA
    bool f16 = false;                 // fp16 q, ckv and kpe (narrow or two-CTA kernel) instead of bf16
    int segment_cost = 0;             // partition cost of a request start, in tiles
    std::vector<int32_t> unit_ptr;
    std::vector<Segment> segments;
    int num_partials = 0;
    int num_split = 0;                // requests cut into several pieces
    PlanLayout layout;
};

constexpr int kMaxQoLen = 64;

// Returns 0 on success, 1 invalid argument, 2 unsupported.
int build_plan(const int32_t* kv_indptr, const int32_t* kv_last_page_len, int batch, int qo_len, bool causal,
               int h_q, int page_size, int num_sms, int kv_dtype, int out_dtype, PlanData* out);

// Heads handled by one CTA for a given h_q and cache type (0 if unsupported): bf16 cache, all
// of them (the narrow-head kernel for h_q <= 32, the two-CTA kernel for 64/128); e4m3 cache, 16
// (the tcgen05 e4m3 kernel, h_q / 16 CTAs per unit); INT8 cache, h_q up to 32 (the 8-bit
// warp-MMA kernel, h_q / 32 CTAs per unit above).
int heads_per_cta_for(int h_q, int kv_dtype);

}  // namespace mla
