// Balanced split-KV scheduler (host only).
//
// FlashMLA PR #233 lists a "balanced scheduler" and a "deterministic combine"
// for its decode kernel without spelling out the partition; the reading used
// here is the plainest one that balances SMs: lay every request's tokens end
// to end in request order, cut the sequence into tiles of the kernel's tile size
// (32 tokens for the bf16 cache with 16/32 heads, 128 otherwise; a request's last tile may
// be short), and cut the sequence into U contiguous ranges, one per CTA slot, that
// minimise the largest range cost.  A tile costs 1; every segment of a range after its
// first also costs the kernel's segment cost in tiles, because a CTA that moves on to
// another request pays a second segment prologue and epilogue (query load, merge of its
// warp groups, output or partial write).  A request whose tiles land in more than one slot becomes
// several split pieces, each writing a partial (out, lse); the CTA finishing the
// last piece merges them in slot order.
//
// With qo_len query tokens per request (several new tokens decoded at once), every
// (request, query token) pair is a query row of its own, laid out in order on the same
// axis: row b * qo_len + j reads request b's pages, over its first L_b tokens, or, causal
// within the new tokens, over its first L_b - (qo_len - 1 - j) (the new tokens being the
// last qo_len of the cache).  Each row streams its pages itself.
#include "plan.h"

#include <algorithm>

namespace mla {

namespace {
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace

int heads_per_cta_for(int h_q, int kv_dtype) {
    const bool ok = h_q == 16 || h_q == 32 || h_q == 64 || h_q == 128;
    // e4m3 cache: the tcgen05 e4m3 kernel, 16 heads per CTA (h_q / 16 CTAs per unit, each streaming
    // the unit's pages, the repeats mostly from L2).  (The 8-bit warp-MMA kernel also serves e4m3
    // codes; at 16 heads it measured 273 us against this kernel's 175 us on 64 x 16384 tokens.)
    if (kv_dtype == 1) return ok ? 16 : 0;
    // INT8 cache: the 8-bit narrow kernel, 32 heads per CTA above 32 heads
    if (kv_dtype == 2) return ok ? (h_q <= 32 ? h_q : 32) : 0;
    switch (h_q) {
        case 16:
        case 32:
        case 64:
        case 128: return h_q;
        default: return 0;
    }
}

int build_plan(const int32_t* kv_indptr, const int32_t* kv_last_page_len, int batch, int qo_len, bool causal,
               int h_q, int page_size, int num_sms, int kv_dtype, int out_dtype, PlanData* out) {
    if (!kv_indptr || !kv_last_page_len || !out || batch < 1 || num_sms < 1) return 1;
    if (kv_dtype < 0 || kv_dtype > 3) return 1;
    if (out_dtype != 0 && out_dtype != 1) return 1;
    if (qo_len < 1 || qo_len > kMaxQoLen) return 1;
    if (static_cast<int64_t>(batch) * qo_len * 128 >= (int64_t(1) << 31)) return 1;
    if (page_size != 16 && page_size != 32 && page_size != 64) return 2;
    const int hg = heads_per_cta_for(h_q, kv_dtype);
    if (hg == 0) return 2;
    if (kv_indptr[0] != 0) return 1;

    const bool eight = kv_dtype == 1 || kv_dtype == 2;
    const bool narrow = h_q <= 32 && !eight;
    const bool narrow8 = kv_dtype == 2;
    const bool e4m3 = kv_dtype == 1 && !narrow8;
    const int tile_tok = (narrow || narrow8) ? kNarrowTileTokens : kTileTokens;
    const int rows = batch * qo_len;
    std::vector<int64_t> len(rows), tiles(rows);
    int64_t total_tiles = 0;
    for (int b = 0; b < batch; ++b) {
        int64_t n = static_cast<int64_t>(kv_indptr[b + 1]) - kv_indptr[b];
        if (n < 0) return 1;
        int64_t L = 0;
        if (n > 0) {
            int last = kv_last_page_len[b];
            if (last < 1 || last > page_size) return 1;
            L = (n - 1) * page_size + last;
            if (L > (int64_t(1) << 30)) return 1;
        }
        for (int j = 0; j < qo_len; ++j) {
            const int r = b * qo_len + j;
            len[r] = causal ? std::max<int64_t>(0, L - (qo_len - 1 - j)) : L;
            tiles[r] = (len[r] + tile_tok - 1) / tile_tok;
            total_tiles += tiles[r];
        }
    }

    PlanData p;
    p.batch = batch;
    p.qo_len = qo_len;
    p.causal = causal;
    p.out_dtype = out_dtype;
    p.rows = rows;
    p.h_q = h_q;
    p.page_size = page_size;
    p.num_sms = num_sms;
    p.kv_dtype = kv_dtype;
    p.heads_per_cta = hg;
    p.head_groups = h_q / hg;
    p.tile_tokens = tile_tok;
    p.narrow = narrow;
    p.pair = h_q >= 64 && !eight;
    p.e4m3 = e4m3;
    p.narrow8 = narrow8;
    p.f16 = kv_dtype == 3;
    const int ctas_per_unit = p.head_groups * (p.pair ? 2 : 1);
    int64_t units = std::max(1, num_sms / ctas_per_unit);
    units = std::min<int64_t>(units, std::max<int64_t>(total_tiles, 1));
    p.num_units = static_cast<int>(units);
    p.segment_cost = (narrow || narrow8) ? kNarrowSegmentCost : kSegmentCost;

    // A unit's cost is its tiles plus segment_cost for every segment after its first (each
    // further segment pays a query load, an epilogue and a partial write or a merge).  fill(T)
    // walks the rows in order and gives each unit tiles until one more segment would pass T;
    // it returns the number of units used.  Giving a unit more tiles never adds to a later
    // unit's cost, so the smallest T with fill(T) <= units is the smallest maximum cost any
    // contiguous partition reaches.
    const int64_t c = p.segment_cost;
    std::vector<std::vector<Segment>> per_unit;
    std::vector<int> pieces(rows, 0);
    int64_t fill_max_pieces = 0;   // (set by fill) the most pieces any request was cut into
    auto fill = [&](int64_t T, bool record) -> int64_t {
        int64_t used = 0, cost = 0, segs = 0;
        fill_max_pieces = 0;
        for (int b = 0; b < rows; ++b) {
            int64_t np = 0;
            for (int64_t t = 0; t < tiles[b];) {
                int64_t room = used == 0 ? 0 : T - cost - (segs > 0 ? c : 0);
                if (room < 1) {
                    ++used;
                    cost = 0;
                    segs = 0;
                    room = T;
                    if (record) per_unit.emplace_back();
                }
                const int64_t k = std::min(tiles[b] - t, room);
                if (record) {
                    Segment sg{};
                    sg.b = b;
                    sg.kv = b / qo_len;
                    sg.t_begin = static_cast<int32_t>(t * tile_tok);
                    sg.t_end = static_cast<int32_t>(std::min<int64_t>((t + k) * tile_tok, len[b]));
                    sg.slot = -1;
                    sg.item = -1;
                    per_unit.back().push_back(sg);
                    ++pieces[b];
                }
                cost += k + (segs > 0 ? c : 0);
                ++segs;
                t += k;
                ++np;
            }
            fill_max_pieces = std::max(fill_max_pieces, np);
        }
        return used;
    };
    auto min_bound = [&](int64_t U) {   // the smallest T with fill(T) <= U
        int64_t lo = 1, hi = total_tiles + c * rows + 1;   // fill(hi) is 1 (or 0 with no tiles)
        while (lo < hi) {
            const int64_t mid = lo + (hi - lo) / 2;
            if (fill(mid, false) <= U)
                hi = mid;
            else
                lo = mid + 1;
        }
        return lo;
    };
    // A split request is merged by its last piece after every piece is done, reading the
    // others' partials: about merge_q / 4 tiles' time per piece.  With few
    // requests, cutting them over every SM makes that merge the longest step (one 4096-token
    // request over 128 SMs: 128 pieces), so the plan weighs a unit count U by
    // bound(U) + merge cost x (most pieces of a request at U) over U = units * k / 16 and takes
    // the cheapest (the full count on ties).
    const double merge_q = (e4m3 ? kMergeCostQuarterTilesE4m3 : kMergeCostQuarterTiles) / 4.0;
    int64_t best_T = min_bound(units), best_U = units;
    double best_score = static_cast<double>(best_T) + (fill_max_pieces > 1 ? merge_q * fill_max_pieces : 0.0);
    for (int k = 15; k >= 1; --k) {
        const int64_t U = std::max<int64_t>(1, units * k / 16);
        if (U >= best_U && U != 1) continue;
        const int64_t T = min_bound(U);
        const double score = static_cast<double>(T) + (fill_max_pieces > 1 ? merge_q * fill_max_pieces : 0.0);
        if (score < best_score) {
            best_score = score;
            best_T = T;
            best_U = U;
        }
    }
    fill(best_T, true);
    // the units the fill used (the cost bound may leave the last ones without tiles)
    units = std::max<int64_t>(1, static_cast<int64_t>(per_unit.size()));
    per_unit.resize(static_cast<size_t>(units));
    p.num_units = static_cast<int>(units);
    // partial slots: a split request's pieces get consecutive slots in token order
    std::vector<int> slot_begin(rows, -1);
    int next_slot = 0;
    for (int b = 0; b < rows; ++b) {
        if (pieces[b] > 1) {
            slot_begin[b] = next_slot;
            next_slot += pieces[b];
        }
    }
    // split requests get an arrival counter each; empty requests become zero-length
    // segments spread round-robin over the units (their CTA writes out = 0, lse = -inf)
    std::vector<int> item_of(rows, -1);
    int next_item = 0;
    for (int b = 0; b < rows; ++b)
        if (pieces[b] > 1) item_of[b] = next_item++;
    int rr = 0;
    for (int b = 0; b < rows; ++b)
        if (pieces[b] == 0) {
            per_unit[rr % units].push_back(Segment{b, 0, 0, -1, -1, 0, 0, b / qo_len});
            ++rr;
        }
    std::vector<int> used(rows, 0);
    p.unit_ptr.push_back(0);
    for (int64_t v = 0; v < units; ++v) {
        for (Segment s : per_unit[v]) {
            if (pieces[s.b] > 1) {
                s.slot = slot_begin[s.b] + used[s.b]++;
                s.item = item_of[s.b];
                s.slot_begin = slot_begin[s.b];
                s.n_slots = pieces[s.b];
            }
            p.segments.push_back(s);
        }
        p.unit_ptr.push_back(static_cast<int32_t>(p.segments.size()));
    }
    p.num_partials = next_slot;
    p.num_split = next_item;

    PlanLayout& L = p.layout;
    L.off_status = 0;
    L.off_unit_ptr = 256;
    L.off_segments = align_up(L.off_unit_ptr + sizeof(int32_t) * p.unit_ptr.size(), 16);
    L.off_counters = align_up(L.off_segments + sizeof(Segment) * p.segments.size(), 16);
    L.header_bytes = align_up(L.off_counters + 2 * sizeof(int32_t) * size_t(p.num_split) * (h_q / 16), 256);
    L.off_part_lse = L.header_bytes;
    L.off_part_o = align_up(L.off_part_lse + sizeof(float) * size_t(p.num_partials) * h_q, 256);
    L.total_bytes = align_up(L.off_part_o + sizeof(float) * size_t(p.num_partials) * h_q * kDimCkv, 256);

    *out = std::move(p);
    return 0;
}

}  // namespace mla
