"""Properties of the host split-KV plan (no GPU): every token of every request
is covered exactly once, cuts fall on the kernel's tile boundaries (32 tokens
for 16/32 heads, 128 for 64/128), the cost per CTA slot (tiles plus a fixed
cost per request start) is balanced, split pieces get consecutive partial
slots in token order, and the plan is a deterministic function of its
inputs."""
import random

import numpy as np
import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
from mla_paged_kv_decode_gb300 import build as lib_build



@pytest.fixture(scope="module", autouse=True)
def _lib():
    if lib_build.needs_build():
        lib_build.build()
    mla.load()


def _lens_to_arrays(lens, P):
    n = [(L + P - 1) // P for L in lens]
    indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    last = np.array([L - (k - 1) * P if k > 0 else 0 for L, k in zip(lens, n)], dtype=np.int32)
    return indptr, last


def _fits(row_tiles, T, c, units):
    """Whether the rows' tiles, in order, split into at most `units` contiguous ranges of cost
    <= T (a range's cost: its tiles plus c per segment after its first).  Filling each range as
    far as it goes is optimal: a range that takes more leaves the next ones less to carry and
    no more segments."""
    if T < 1:
        return False
    used, cost, segs = 0, 0, 0
    for n in row_tiles:
        left = n
        while left:
            room = T - cost - (c if segs else 0) if used else 0
            if room < 1:
                used, cost, segs, room = used + 1, 0, 0, T
            k = min(left, room)
            cost += k + (c if segs else 0)
            segs += 1
            left -= k
    return used <= units


def _check_plan(lens, h_q, P, sms, kv_dtype=mla.MLA_KV_BF16):
    bf16 = kv_dtype == mla.MLA_KV_BF16
    # the kernels: bf16 cache -- warp-MMA kernel up to 32 heads, two-CTA tcgen05 kernel above;
    # e4m3 cache -- the tcgen05 e4m3 kernel (16 heads a CTA); INT8 cache -- the 8-bit warp-MMA
    # kernel (up to 32 heads a CTA).  The tile is 32 tokens for the warp-MMA kernels, 128 for the
    # tcgen05 ones.
    tcgen05 = kv_dtype == mla.MLA_KV_FP8_E4M3 or (h_q >= 64 and bf16)
    TILE = 128 if tcgen05 else 32
    if bf16:
        want_hg = h_q
    elif kv_dtype == mla.MLA_KV_FP8_E4M3:
        want_hg = 16
    else:
        want_hg = min(h_q, 32)
    indptr, last = _lens_to_arrays(lens, P)
    plan = mla.mla_decode_plan(torch.from_numpy(indptr), torch.from_numpy(last), len(lens), h_q, P, sms, kv_dtype)
    segs, uptr = mla.mla_plan_get_segments(plan)
    hg = mla.mla_plan_heads_per_cta(plan)
    assert hg == want_hg
    groups = h_q // hg
    units = len(uptr) - 1
    assert units == mla.mla_plan_num_units(plan)
    pair = 2 if (h_q >= 64 and bf16) else 1   # bf16 64/128 heads: a cluster of two CTAs per unit
    assert mla.mla_plan_num_ctas(plan) == units * groups * pair
    assert units <= max(1, sms // (groups * pair))
    # coverage: each request's tokens exactly once, pieces in token order
    covered = {b: [] for b in range(len(lens))}
    empties = []
    for b, t0, t1, slot in segs:
        if lens[b] == 0:
            assert t0 == 0 and t1 == 0 and slot == -1   # zero-length segment: write out = 0, lse = -inf
            empties.append(int(b))
            continue
        assert 0 <= t0 < t1 <= lens[b]
        assert t0 % TILE == 0 and (t1 % TILE == 0 or t1 == lens[b])
        covered[b].append((t0, t1, slot))
    assert sorted(empties) == [b for b, L in enumerate(lens) if L == 0], "each empty request exactly once"
    order = [int(b) for b, t0, t1, _ in segs if t1 > t0]
    assert order == sorted(order), "segments follow request order"
    n_split = 0
    for b, L in enumerate(lens):
        pieces = sorted(covered[b])
        if L == 0:
            assert pieces == []
            continue
        assert pieces[0][0] == 0 and pieces[-1][1] == L
        for (a0, a1, _), (b0, b1, _) in zip(pieces, pieces[1:]):
            assert a1 == b0
        if len(pieces) == 1:
            assert pieces[0][2] == -1
        else:
            slots = [p[2] for p in pieces]
            assert slots == list(range(slots[0], slots[0] + len(slots)))
            n_split += len(pieces)
    assert mla.mla_plan_num_partials(plan) == n_split
    # balance: a unit's cost is its tiles plus c for every segment after its first.  The plan's
    # largest unit cost must be the smallest any contiguous partition of the request order into
    # at most the units it uses reaches: no partition with a smaller maximum exists (_fits, an
    # exhaustive-by-greedy feasibility test), and every unit holds tiles.  (The plan may use
    # fewer units than the GPU has, when cutting few requests over every SM would make their
    # merges the longest step.)
    c = mla.mla_plan_segment_cost_tiles(plan)
    assert c >= 0
    tiles, cost = [], []
    for u in range(units):
        s = [x for x in segs[uptr[u]:uptr[u + 1]] if x[2] > x[1]]
        nt = sum((int(t1) - int(t0) + TILE - 1) // TILE for _, t0, t1, _ in s)
        tiles.append(nt)
        cost.append(nt + c * max(0, len(s) - 1))
    row_tiles = [(L + TILE - 1) // TILE for L in lens]
    total = sum(row_tiles)
    assert sum(tiles) == total
    if total:
        assert min(tiles) >= 1
        assert not _fits([t for t in row_tiles if t], max(cost) - 1, c, units), (max(cost), c)
    # workspace holds every partial
    assert plan.workspace_bytes >= n_split * h_q * (512 + 1) * 4
    return segs, uptr


def test_uniform_batch():
    _check_plan([4096] * 64, 16, 64, 152)


def test_compute_shape_groups():
    segs, uptr = _check_plan([8192] * 128, 128, 64, 152)
    assert len(uptr) - 1 <= 152 // 2          # one unit per pair of SMs
    segs, uptr = _check_plan([8192] * 128, 64, 64, 152)
    assert len(uptr) - 1 <= 152 // 2          # 64 heads: the same two-CTA unit


def test_tiny_and_edge_lengths():
    _check_plan([1, 17, 64, 203], 16, 16, 152)
    _check_plan([0, 5, 0, 129], 32, 32, 3)
    _check_plan([0], 16, 16, 152)
    _check_plan([128 * 40], 64, 64, 152)
    _check_plan([1] * 300, 16, 16, 152)


def test_random_plans():
    rng = random.Random(1234)
    for _ in range(60):
        B = rng.randint(1, 80)
        lens = [rng.choice([0, 1, rng.randint(1, 300), rng.randint(1, 20000)]) for _ in range(B)]
        _check_plan(lens, rng.choice([16, 32, 64, 128]), rng.choice([16, 32, 64]), rng.choice([1, 7, 64, 152]))


def test_e4m3_plans():
    """The e4m3 cache runs on the tcgen05 kernel: 128-token tiles, 16 heads per CTA."""
    segs, uptr = _check_plan([16384] * 64, 16, 64, 152, mla.MLA_KV_FP8_E4M3)
    assert len(uptr) - 1 <= 152
    segs, uptr = _check_plan([4096] * 8, 32, 64, 152, mla.MLA_KV_FP8_E4M3)
    assert len(uptr) - 1 <= 152 // 2          # two 16-head CTAs per unit
    rng = random.Random(99)
    for _ in range(20):
        B = rng.randint(1, 60)
        lens = [rng.choice([0, 1, rng.randint(1, 300), rng.randint(1, 20000)]) for _ in range(B)]
        _check_plan(lens, rng.choice([16, 32]), rng.choice([16, 32, 64]), rng.choice([1, 7, 64, 152]),
                    mla.MLA_KV_FP8_E4M3)
    for h_q, units in ((64, 38), (128, 19)):  # wider heads: h_q / 16 CTAs of 16 heads per unit
        segs, uptr = _check_plan([8192] * 16, h_q, 64, 152, mla.MLA_KV_FP8_E4M3)
        assert len(uptr) - 1 <= units


def test_plan_is_deterministic():
    lens = [random.Random(7).randint(1, 32768) for _ in range(256)]
    a = _check_plan(lens, 128, 16, 152)
    b = _check_plan(lens, 128, 16, 152)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_request_starts_cost_tiles():
    """Units that cross into another request get fewer tiles than units inside one."""
    segs, uptr = _check_plan([4096] * 64, 16, 64, 152)
    TILE = 32
    indptr, last = _lens_to_arrays([4096] * 64, 64)
    plan = mla.mla_decode_plan(torch.from_numpy(indptr), torch.from_numpy(last), 64, 16, 64, 152)
    c = mla.mla_plan_segment_cost_tiles(plan)
    inside, crossing = [], []
    for u in range(len(uptr) - 1):
        s = segs[uptr[u]:uptr[u + 1]]
        nt = sum((int(t1) - int(t0) + TILE - 1) // TILE for _, t0, t1, _ in s)
        (crossing if len(s) > 1 else inside).append(nt)
    assert inside and crossing
    # a unit ending inside the next request's start cost also has fewer tiles, so compare means
    assert sum(inside) / len(inside) - sum(crossing) / len(crossing) >= c / 2


@pytest.mark.parametrize("qo_len,causal,h_q,kv_dtype", [(2, True, 16, mla.MLA_KV_BF16), (3, True, 128, mla.MLA_KV_BF16),
                                                         (3, False, 64, mla.MLA_KV_BF16), (4, True, 16, mla.MLA_KV_FP8_E4M3)])
def test_query_rows_plan(qo_len, causal, h_q, kv_dtype):
    """Several query tokens per request: row b * qo_len + j covers exactly the first
    max(0, L_b - (qo_len - 1 - j)) tokens (causal) or all L_b, once, and nothing else."""
    rng = random.Random(7 + qo_len)
    P = 16
    lens = [rng.choice([0, 1, 2, rng.randint(3, 300), rng.randint(300, 5000)]) for _ in range(37)]
    indptr, last = _lens_to_arrays(lens, P)
    plan = mla.mla_decode_plan_ex(torch.from_numpy(indptr), torch.from_numpy(last), len(lens), qo_len, causal, h_q,
                                  P, 152, kv_dtype, mla.MLA_OUT_BF16)
    assert mla.mla_plan_num_rows(plan) == len(lens) * qo_len
    segs, uptr = mla.mla_plan_get_segments(plan)
    covered = {}
    for r, t0, t1, _ in segs:
        covered.setdefault(int(r), []).append((int(t0), int(t1)))
    for b, L in enumerate(lens):
        for j in range(qo_len):
            r = b * qo_len + j
            Lr = max(0, L - (qo_len - 1 - j)) if causal else L
            pieces = sorted(covered.get(r, []))
            assert pieces, f"row {r} missing"
            if Lr == 0:
                assert pieces == [(0, 0)]
                continue
            assert pieces[0][0] == 0 and pieces[-1][1] == Lr
            for (a0, a1), (b0, b1) in zip(pieces, pieces[1:]):
                assert a1 == b0
    assert set(covered) == set(range(len(lens) * qo_len))


def test_query_rows_argument_checks():
    indptr, last = _lens_to_arrays([5, 9], 16)
    ip, lp = torch.from_numpy(indptr), torch.from_numpy(last)
    for qo_len in (0, 65):
        with pytest.raises(mla.MLAError):
            mla.mla_decode_plan_ex(ip, lp, 2, qo_len, True, 16, 16, 152)
    with pytest.raises(mla.MLAError):
        mla.mla_decode_plan_ex(ip, lp, 2, 2, True, 16, 16, 152, out_dtype=2)
    # qo_len 1 with fp32 output is mla_decode_plan itself
    a = mla.mla_decode_plan(ip, lp, 2, 16, 16, 152)
    b = mla.mla_decode_plan_ex(ip, lp, 2, 1, True, 16, 16, 152)
    sa, ua = mla.mla_plan_get_segments(a)
    sb, ub = mla.mla_plan_get_segments(b)
    assert np.array_equal(sa, sb) and np.array_equal(ua, ub)


def test_query_rows_plan_fuzz():
    """Random batches, heads, page sizes, cache types and qo_len: every row's causal prefix is
    covered exactly once, in order, with consecutive partial slots for split rows."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=60, deadline=None)
    @hyp.given(lens=st.lists(st.integers(0, 3000), min_size=1, max_size=24), qo_len=st.integers(1, 5),
               causal=st.booleans(), h_q=st.sampled_from([16, 32, 64, 128]), P=st.sampled_from([16, 32, 64]),
               fp8=st.booleans(), sms=st.sampled_from([1, 7, 152]))
    def check(lens, qo_len, causal, h_q, P, fp8, sms):
        indptr, last = _lens_to_arrays(lens, P)
        kvd = mla.MLA_KV_FP8_E4M3 if fp8 else mla.MLA_KV_BF16
        plan = mla.mla_decode_plan_ex(torch.from_numpy(indptr), torch.from_numpy(last), len(lens), qo_len, causal,
                                      h_q, P, sms, kvd)
        segs, uptr = mla.mla_plan_get_segments(plan)
        assert uptr[0] == 0 and uptr[-1] == len(segs) and all(np.diff(uptr) >= 0)
        per_row = {}
        for r, t0, t1, slot in segs:
            per_row.setdefault(int(r), []).append((int(t0), int(t1), int(slot)))
        n_split = 0
        for b, L in enumerate(lens):
            for j in range(qo_len):
                r = b * qo_len + j
                Lr = max(0, L - (qo_len - 1 - j)) if causal else L
                pieces = sorted(per_row.pop(r))
                if Lr == 0:
                    assert pieces == [(0, 0, -1)]
                    continue
                assert pieces[0][0] == 0 and pieces[-1][1] == Lr
                assert all(a[1] == c[0] for a, c in zip(pieces, pieces[1:]))
                if len(pieces) > 1:
                    slots = [p[2] for p in pieces]
                    assert slots == list(range(slots[0], slots[0] + len(slots)))
                    n_split += len(pieces)
                else:
                    assert pieces[0][2] == -1
        assert not per_row
        assert mla.mla_plan_num_partials(plan) == n_split

    check()


def test_int8_plans():
    """The INT8 cache runs on the 8-bit warp-MMA kernel: 32-token tiles, up to 32 heads per CTA
    (64 and 128 heads: 2 or 4 CTAs per unit, each streaming the unit's pages)."""
    segs, uptr = _check_plan([16384] * 64, 16, 64, 152, mla.MLA_KV_INT8)
    assert len(uptr) - 1 <= 152
    for h_q, units in ((32, 152), (64, 76), (128, 38)):
        segs, uptr = _check_plan([4096] * 16, h_q, 64, 152, mla.MLA_KV_INT8)
        assert len(uptr) - 1 <= units
    rng = random.Random(7)
    for _ in range(20):
        B = rng.randint(1, 60)
        lens = [rng.choice([0, 1, rng.randint(1, 300), rng.randint(1, 20000)]) for _ in range(B)]
        _check_plan(lens, rng.choice([16, 32, 64, 128]), rng.choice([16, 32, 64]), rng.choice([1, 7, 64, 152]),
                    mla.MLA_KV_INT8)


def test_few_long_requests_are_not_cut_over_every_sm():
    """One 4096-token request at 16 heads is 128 tiles: cut over 128 SMs, its last piece would
    merge 128 partials.  The plan weighs the merge (about a tile per piece) against the
    streaming time and cuts it into far fewer pieces; a full batch still uses every SM."""
    for lens, h_q, kv in (([4096], 16, mla.MLA_KV_BF16), ([32768], 128, mla.MLA_KV_BF16),
                          ([4096], 16, mla.MLA_KV_FP8_E4M3)):
        segs, uptr = _check_plan(lens, h_q, 64, 152, kv)
        pieces = sum(1 for b, t0, t1, _ in segs if t1 > t0)
        tile = 32 if (h_q <= 32 and kv == mla.MLA_KV_BF16) else 128
        tiles = (lens[0] + tile - 1) // tile
        assert 2 <= pieces <= 2 * int(tiles ** 0.5) + 2, (lens, h_q, pieces)
    segs, uptr = _check_plan([4096] * 64, 16, 64, 152)
    assert len(uptr) - 1 >= 148
