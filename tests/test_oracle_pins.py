"""Pins for the fp64 oracle: each compares it with something other than itself.

The pages print no worked numeric example of MLA decode, so the oracle is
pinned by hand-derived closed forms (tests/golden), a second independent
statement (torch fp64 brute force with library softmax), invariants of the
mathematics (softmax shift/scale, page placement, split + merge), and library
routines for the e4m3 codec.  ``test_planted_mistakes_are_caught`` builds
copies of the oracle with a deliberate mistake and checks these pins fail.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.brute import brute_force, brute_force_rows
from workloads import WORKLOADS, make_inputs, quantize_e4m3_per_token, quantize_int8_per_token, query_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CONSTS = {"ln2": math.log(2.0), "ln3": math.log(3.0), "ln4": math.log(4.0), "ln1.5": math.log(1.5)}


def _val(v):
    return CONSTS[v] if isinstance(v, str) else float(v)


def _load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    H, P, N = g["h_q"], g["page_size"], g["num_pages"]
    B = len(g["kv_indptr"]) - 1
    q_nope = torch.zeros(B, H, 512)
    q_pe = torch.zeros(B, H, 64)
    for h, ents in g["q_nope_nonzero"].items():
        for d, v in ents:
            q_nope[0, int(h), d] = v
    for h, ents in g["q_pe_nonzero"].items():
        for d, v in ents:
            q_pe[0, int(h), d] = v
    ckv = torch.zeros(N, P, 512)
    kpe = torch.zeros(N, P, 64)
    for pg, ents in g["ckv_nonzero"].items():
        for s, d, v in ents:
            ckv[int(pg[4:]), s, d] = v
    for pg, ents in g["kpe_nonzero"].items():
        for s, d, v in ents:
            kpe[int(pg[4:]), s, d] = v
    for pg in g.get("nan_pages", []):
        ckv[pg] = float("nan")
        kpe[pg] = float("nan")
    exp_out = torch.zeros(B, H, 512, dtype=torch.float64)
    for h, ents in g["expected_out_nonzero"].items():
        for d, v in ents:
            exp_out[0, int(h), d] = v
    exp_lse = torch.tensor([[_val(v) for v in row] for row in g["expected_lse"]], dtype=torch.float64)
    args = (q_nope.bfloat16(), q_pe.bfloat16(), ckv.bfloat16(), kpe.bfloat16(),
            torch.tensor(g["kv_indices"], dtype=torch.int32), torch.tensor(g["kv_indptr"], dtype=torch.int32),
            torch.tensor(g["kv_last_page_len"], dtype=torch.int32), _val(g["sm_scale"]))
    return args, exp_out, exp_lse, g["tolerance"]


def _tiny_args(inp, sm_scale=None):
    return (inp.q_nope, inp.q_pe, inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr, inp.kv_last_page_len,
            inp.sm_scale if sm_scale is None else sm_scale)


def _small(seed=11, kv_lens=(1, 5, 33, 70), H=4, P=16, pool=None):
    return make_inputs(WORKLOADS["tiny"], kv_lens=list(kv_lens), batch=len(kv_lens), h_q=H, page_size=P,
                       pool_pages=pool, seed=seed)


# ---------------------------------------------------------------- golden, hand-derived

@pytest.mark.parametrize("name", ["two_token_ln3.json", "gather_kpe_sign.json"])
def test_golden_closed_form(name, lib=None):
    args, exp_out, exp_lse, tol = _load_golden(name)
    out, lse = oracle.mla_decode(*args, lib=lib)
    assert torch.allclose(out, exp_out, atol=tol, rtol=0), (out[..., :4], exp_out[..., :4])
    assert torch.allclose(lse, exp_lse, atol=tol, rtol=0), (lse, exp_lse)


# ---------------------------------------------------------------- brute force (library softmax)

@pytest.mark.parametrize("case", ["tiny", "small_p16", "small_p1", "small_p64"])
def test_matches_brute_force(case, lib=None):
    if case == "tiny":
        inp = make_inputs(WORKLOADS["tiny"])
    elif case == "small_p16":
        inp = _small()
    elif case == "small_p1":
        inp = _small(seed=12, kv_lens=(3, 1, 9), H=3, P=1, pool=20)
    else:
        inp = _small(seed=13, kv_lens=(64, 65, 130), H=2, P=64, pool=6)
    out, lse = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    bo, bl = brute_force(*_tiny_args(inp))
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    assert (out - bo).abs().max().item() <= 1e-12
    assert (lse - bl).abs().max().item() <= 1e-12


def test_matches_brute_force_fp8(lib=None):
    inp = make_inputs(WORKLOADS["fp8"], kv_lens=[5, 70, 128], batch=3, h_q=4, page_size=64, seed=21)
    out, lse = oracle.mla_decode(*_tiny_args(inp), ckv_scale=inp.ckv_scale, lib=lib)
    bo, bl = brute_force(*_tiny_args(inp), ckv_scale=inp.ckv_scale)
    assert (out - bo).abs().max().item() <= 1e-12
    assert (lse - bl).abs().max().item() <= 1e-12


# ---------------------------------------------------------------- closed forms and invariants

def test_single_token_returns_its_value_row(lib=None):
    """L = 1: softmax of one score is 1, so out is that token's ckv row exactly."""
    inp = make_inputs(WORKLOADS["tiny"])
    out, lse = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    pg = int(inp.kv_indices[inp.kv_indptr[0]])
    v0 = inp.ckv[pg, 0].to(torch.float64)
    assert inp.kv_lens[0] == 1
    assert torch.equal(out[0], v0.expand_as(out[0]))
    bo, bl = brute_force(*_tiny_args(inp))
    assert torch.equal(lse[0], bl[0]) or (lse[0] - bl[0]).abs().max() < 1e-13


def test_zero_scale_gives_mean_and_log_length(lib=None):
    """sm_scale = 0: every score is 0, out = mean of the ckv rows, lse = ln L."""
    inp = _small(seed=5, kv_lens=(7, 40))
    out, lse = oracle.mla_decode(*_tiny_args(inp, sm_scale=0.0), lib=lib)
    for b in range(inp.batch):
        L = int(inp.kv_lens[b])
        pages = inp.kv_indices[inp.kv_indptr[b]:inp.kv_indptr[b + 1]].tolist()
        rows = np.stack([inp.ckv[pages[t // 16], t % 16].double().numpy() for t in range(L)])
        mean = rows.mean(axis=0)
        assert np.abs(out[b].numpy() - mean[None, :]).max() < 1e-12
        assert np.abs(lse[b].numpy() - math.log(L)).max() < 1e-12


def test_identical_keys_give_mean_of_values(lib=None):
    """q_nope = 0 and identical kpe rows: all scores equal, out = mean(ckv rows), lse = x + ln L."""
    inp = _small(seed=6, kv_lens=(9, 31), H=3)
    inp.q_nope.zero_()
    inp.kpe.copy_(inp.kpe[0, 0].expand_as(inp.kpe))
    out, lse = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    x = inp.sm_scale * (inp.q_pe.double() @ inp.kpe[0, 0].double())   # [B, H]
    for b in range(inp.batch):
        L = int(inp.kv_lens[b])
        pages = inp.kv_indices[inp.kv_indptr[b]:inp.kv_indptr[b + 1]].tolist()
        mean = np.stack([inp.ckv[pages[t // 16], t % 16].double().numpy() for t in range(L)]).mean(0)
        assert np.abs(out[b].numpy() - mean[None, :]).max() < 1e-12
        assert (lse[b] - (x[b] + math.log(L))).abs().max() < 1e-12


def test_score_shift_moves_only_lse(lib=None):
    """Adding c to every token's kpe[0] with q_pe = e_0 shifts all scores by sm_scale*c:
    out is unchanged (softmax shift invariance), lse moves by exactly sm_scale*c."""
    inp = _small(seed=7, kv_lens=(12, 50), H=2)
    inp.q_pe.zero_()
    inp.q_pe[:, :, 0] = 1.0
    inp.kpe[:, :, 0] = 0.0
    out0, lse0 = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    c = 8.0
    inp.kpe[:, :, 0] = c
    out1, lse1 = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    assert (out1 - out0).abs().max() < 1e-12
    assert (lse1 - lse0 - inp.sm_scale * c).abs().max() < 1e-12


def test_dominant_score_selects_one_row(lib=None):
    """Scores spread over ~2000 logits: the largest one takes all the weight, so out is that
    token's ckv row and lse is its score (exp(-1000) underflows to 0 against 1)."""
    inp = _small(seed=15, kv_lens=(37,), H=2)
    inp.q_nope.zero_()
    inp.q_pe.zero_()
    inp.q_pe[:, :, 0] = 1.0
    g = torch.Generator().manual_seed(5)
    vals = (torch.randperm(37, generator=g).float() * 64 - 1024)      # distinct, spaced 64 apart
    pages = inp.kv_indices[inp.kv_indptr[0]:inp.kv_indptr[1]].tolist()
    for t in range(37):
        inp.kpe[pages[t // 16], t % 16, 0] = vals[t]
    sm = 1.0
    out, lse = oracle.mla_decode(*_tiny_args(inp, sm_scale=sm), lib=lib)
    t_star = int(torch.argmax(vals))
    v = inp.ckv[pages[t_star // 16], t_star % 16].double()
    assert torch.isfinite(out).all()
    assert (out[0] - v).abs().max() < 1e-12
    assert (lse[0] - sm * float(vals[t_star])).abs().max() < 1e-12


def test_query_scale_trade(lib=None):
    """q * 2 with sm_scale / 2 leaves every score, hence the result, unchanged."""
    inp = make_inputs(WORKLOADS["tiny"])
    out0, lse0 = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    args = list(_tiny_args(inp))
    args[0] = (inp.q_nope.float() * 2).bfloat16()
    args[1] = (inp.q_pe.float() * 2).bfloat16()
    args[7] = inp.sm_scale / 2
    out1, lse1 = oracle.mla_decode(*args, lib=lib)
    assert (out1 - out0).abs().max() < 1e-13 and (lse1 - lse0).abs().max() < 1e-13


def test_page_permutation_invariance(lib=None):
    """Moving pages to other physical slots (and remapping kv_indices) changes nothing, bit for bit."""
    inp = make_inputs(WORKLOADS["tiny"])
    out0, lse0 = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(inp.num_pages, generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(inp.num_pages)
    ckv = inp.ckv[perm].contiguous()          # new page i holds old page perm[i]
    kpe = inp.kpe[perm].contiguous()
    idx = inv[inp.kv_indices.long()].to(torch.int32)
    out1, lse1 = oracle.mla_decode(inp.q_nope, inp.q_pe, ckv, kpe, idx, inp.kv_indptr, inp.kv_last_page_len,
                                   inp.sm_scale, lib=lib)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_split_then_merge_equals_unsplit(lib=None):
    inp = _small(seed=8, kv_lens=(203, 77))
    out, lse = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    for b, cuts in [(0, [0, 64, 128, 203]), (0, [0, 1, 203]), (1, [0, 16, 17, 60, 77])]:
        parts = [oracle.mla_decode_range(b, a, c, inp.q_nope, inp.q_pe, inp.ckv, inp.kpe, inp.kv_indices,
                                         inp.kv_indptr, inp.sm_scale, lib=lib) for a, c in zip(cuts, cuts[1:])]
        o, l = oracle.merge(torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]), lib=lib)
        assert (o - out[b]).abs().max() < 1e-12 and (l - lse[b]).abs().max() < 1e-12


def test_merge_closed_forms(lib=None):
    """Equal lse -> plain average, lse + ln 2; an empty (-inf) partial has zero weight."""
    g = torch.Generator().manual_seed(3)
    o = torch.randn(2, 3, 8, generator=g, dtype=torch.float64)
    s = torch.tensor([[0.5, -1.0, 2.0]] * 2, dtype=torch.float64)
    out, lse = oracle.merge(o, s, lib=lib)
    assert (out - o.mean(0)).abs().max() < 1e-15
    assert (lse - (s[0] + math.log(2))).abs().max() < 1e-15
    s2 = s.clone()
    s2[1] = float("-inf")
    out2, lse2 = oracle.merge(o, s2, lib=lib)
    assert torch.equal(out2, o[0]) and torch.equal(lse2, s[0])


def test_empty_request(lib=None):
    inp = _small(seed=9, kv_lens=(0, 5))
    out, lse = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    assert torch.equal(out[0], torch.zeros_like(out[0]))
    assert torch.isneginf(lse[0]).all()
    assert torch.isfinite(out[1]).all()


def test_nan_padding_never_read(lib=None):
    """Unused slots and pages are NaN in every generated pool; results stay finite and
    equal to a run where they are zero instead."""
    inp = _small(seed=10, kv_lens=(3, 17, 33), pool=12)
    assert torch.isnan(inp.ckv.float()).any()
    out0, lse0 = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    assert torch.isfinite(out0).all() and torch.isfinite(lse0).all()
    ckv = torch.nan_to_num(inp.ckv.float(), nan=0.0).bfloat16()
    kpe = torch.nan_to_num(inp.kpe.float(), nan=0.0).bfloat16()
    out1, lse1 = oracle.mla_decode(inp.q_nope, inp.q_pe, ckv, kpe, inp.kv_indices, inp.kv_indptr,
                                   inp.kv_last_page_len, inp.sm_scale, lib=lib)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


# ---------------------------------------------------------------- 8-bit cache

def test_e4m3_decode_all_codes(lib=None):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes, lib=lib)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan) and nan.sum() == 2
    assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


def test_e4m3_encode_exhaustive_bf16(lib=None):
    """Every finite bf16 bit pattern with |x| <= 448, against torch's float8_e4m3fn cast."""
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).float()
    keep = torch.isfinite(x) & (x.abs() <= 448.0)
    x = x[keep]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = oracle.e4m3_encode(x.double().numpy(), lib=lib)
    assert np.array_equal(mine, ref), np.nonzero(mine != ref)[0][:10]


def test_generator_quantiser_matches_oracle_encoder(lib=None):
    inp = make_inputs(WORKLOADS["fp8"], kv_lens=[40], batch=1, h_q=2, page_size=64, seed=31)
    x = inp.ckv_bf16[inp.kv_indices[0], :40].double()
    s = inp.ckv_scale[inp.kv_indices[0], :40].double()
    enc = oracle.e4m3_encode((x / s[:, None]).clamp(-448, 448).numpy().astype(np.float32).astype(np.float64), lib=lib)
    # torch quantised in fp32 (x / scale in fp32); compare the same fp32 quotient
    q32 = (inp.ckv_bf16[inp.kv_indices[0], :40].float() / inp.ckv_scale[inp.kv_indices[0], :40, None]).clamp(-448, 448)
    enc32 = oracle.e4m3_encode(q32.double().numpy(), lib=lib)
    assert np.array_equal(enc32, inp.ckv[inp.kv_indices[0], :40].numpy().ravel())
    assert enc.shape == enc32.shape


def test_fp8_bytes_per_token():
    """644 B/token (512 e4m3 + 4-byte scale + 128 B bf16 kpe) instead of 1152 (FlashMLA PR #233)."""
    inp = make_inputs(WORKLOADS["fp8"], kv_lens=[64], batch=1, h_q=1, page_size=64, seed=1)
    per_tok = (inp.ckv[0, 0].numel() * inp.ckv.element_size() + inp.ckv_scale[0, 0].element_size()
               + inp.kpe[0, 0].numel() * inp.kpe.element_size())
    assert per_tok == 644
    bf = make_inputs(WORKLOADS["membound"], kv_lens=[64], batch=1, h_q=1, seed=1)
    assert bf.ckv[0, 0].numel() * 2 + bf.kpe[0, 0].numel() * 2 == 1152


def test_fp8_oracle_equals_bf16_oracle_on_exact_codes(lib=None):
    """When scale * e4m3 reproduces the bf16 cache exactly (power-of-two scales, values on the
    e4m3 grid), the 8-bit oracle and the bf16 oracle see identical numbers."""
    inp = _small(seed=14, kv_lens=(20, 45), H=2, P=16)
    g = torch.Generator().manual_seed(4)
    codes = torch.randint(0, 0x7E, inp.ckv.shape, generator=g, dtype=torch.int32).to(torch.uint8)
    codes |= (torch.randint(0, 2, inp.ckv.shape, generator=g, dtype=torch.int32) << 7).to(torch.uint8)
    scale = torch.pow(2.0, torch.randint(-6, 3, inp.ckv.shape[:2], generator=g).float())
    ckv_bf = (codes.view(torch.float8_e4m3fn).float() * scale[..., None]).bfloat16()
    assert torch.equal(ckv_bf.double(), codes.view(torch.float8_e4m3fn).double() * scale[..., None].double())
    o8, l8 = oracle.mla_decode(inp.q_nope, inp.q_pe, codes, inp.kpe, inp.kv_indices, inp.kv_indptr,
                               inp.kv_last_page_len, inp.sm_scale, ckv_scale=scale, lib=lib)
    ob, lb = oracle.mla_decode(inp.q_nope, inp.q_pe, ckv_bf, inp.kpe, inp.kv_indices, inp.kv_indptr,
                               inp.kv_last_page_len, inp.sm_scale, lib=lib)
    assert torch.equal(o8, ob) and torch.equal(l8, lb)


# ---------------------------------------------------------------- the INT8 cache (oracle side)

def test_matches_brute_force_int8(lib=None):
    inp = make_inputs(WORKLOADS["fp8"], kv_lens=[5, 70, 128], batch=3, h_q=4, page_size=64, seed=22, int8=True)
    assert inp.ckv.dtype == torch.int8
    out, lse = oracle.mla_decode(*_tiny_args(inp), ckv_scale=inp.ckv_scale, lib=lib)
    bo, bl = brute_force(*_tiny_args(inp), ckv_scale=inp.ckv_scale)
    assert torch.isfinite(out).all()
    assert (out - bo).abs().max().item() <= 1e-12
    assert (lse - bl).abs().max().item() <= 1e-12


def test_int8_oracle_equals_bf16_oracle_on_exact_codes(lib=None):
    """Power-of-two scales times integer codes in [-127, 127] are exact in bf16: the INT8 oracle
    and the bf16 oracle then see identical numbers (signed codes: a byte read unsigned fails)."""
    inp = _small(seed=15, kv_lens=(20, 45), H=2, P=16)
    g = torch.Generator().manual_seed(6)
    codes = torch.randint(-127, 128, inp.ckv.shape, generator=g, dtype=torch.int32).to(torch.int8)
    scale = torch.pow(2.0, torch.randint(-8, 2, inp.ckv.shape[:2], generator=g).float())
    ckv_bf = (codes.float() * scale[..., None]).bfloat16()
    assert torch.equal(ckv_bf.double(), codes.double() * scale[..., None].double())
    o8, l8 = oracle.mla_decode(inp.q_nope, inp.q_pe, codes, inp.kpe, inp.kv_indices, inp.kv_indptr,
                               inp.kv_last_page_len, inp.sm_scale, ckv_scale=scale, lib=lib)
    ob, lb = oracle.mla_decode(inp.q_nope, inp.q_pe, ckv_bf, inp.kpe, inp.kv_indices, inp.kv_indptr,
                               inp.kv_last_page_len, inp.sm_scale, lib=lib)
    assert torch.equal(o8, ob) and torch.equal(l8, lb)


def test_int8_quantiser_bounds():
    """Codes within [-127, 127], the token's largest magnitude on +-127, every value within half a
    step of scale * code; an all-zero token gets scale 0 and zero codes."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn(6, 16, 512, generator=g).to(torch.bfloat16)
    x[2, 3] = 0
    codes, scale = quantize_int8_per_token(x)
    assert codes.dtype == torch.int8 and codes.abs().max() <= 127
    xf = x.float()
    err = (xf - codes.float() * scale[..., None]).abs()
    assert (err <= scale[..., None] * 0.5 + xf.abs() * 2.0 ** -21).all()   # x / scale and the check round in fp32
    nz = scale > 0
    assert (codes.abs().amax(dim=-1)[nz] == 127).all()
    assert scale[2, 3] == 0 and (codes[2, 3] == 0).all()


def test_int8_cache_is_close_to_the_bf16_cache(lib=None):
    """The INT8 cache approximates the bf16 one it was quantised from (FlashMLA PR #233 reports a
    worst cosine distance of 2.6e-4 for INT8 on synthetic caches)."""
    inp = make_inputs(WORKLOADS["fp8"], kv_lens=[300, 1000, 77], batch=3, h_q=4, page_size=64, seed=23, int8=True)
    o8, _ = oracle.decode_inputs(inp)
    o16, _ = oracle.decode_inputs(inp, use_bf16_cache=True)
    a, b = o8.flatten(), o16.flatten()
    cd = 1 - float(a @ b / (a.norm() * b.norm()))
    assert cd <= 1e-3, cd


# ---------------------------------------------------------------- several query tokens per request

def _rows_args(inp, qn, qp):
    return (qn, qp, inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr, inp.kv_last_page_len, inp.sm_scale)


@pytest.mark.parametrize("qo_len,causal", [(1, True), (3, True), (3, False), (4, True)])
def test_rows_match_masked_brute_force(qo_len, causal):
    """Row b * qo_len + j over its causal prefix (a range of the definition) equals the whole
    request's scores with the later tokens masked to -inf before a library softmax.  Lengths
    0, 1 and 2 leave some causal rows with no token at all."""
    inp = _small(seed=31, kv_lens=(0, 1, 2, 5, 33, 70), H=3, P=16)
    qn, qp = query_rows(inp, qo_len, seed=32)
    out, lse = oracle.mla_decode_rows(*_rows_args(inp, qn, qp), qo_len, causal)
    bo, bl = brute_force_rows(*_rows_args(inp, qn, qp), qo_len, causal)
    assert torch.equal(torch.isinf(lse), torch.isinf(bl))
    fin = torch.isfinite(bl)
    assert (out - bo).abs().max().item() <= 1e-12
    assert (lse[fin] - bl[fin]).abs().max().item() <= 1e-12
    # the rows left with no token: out 0, lse -inf
    if causal and qo_len > 1:
        assert torch.isinf(lse[1 * qo_len]).all() and (out[1 * qo_len] == 0).all()   # L = 1, j = 0


def test_rows_with_one_token_per_request_equal_decode():
    inp = _small(seed=33)
    out, lse = oracle.mla_decode_rows(*_rows_args(inp, inp.q_nope, inp.q_pe), 1, True)
    o1, l1 = oracle.mla_decode(*_tiny_args(inp))
    assert (out - o1).abs().max().item() <= 1e-13
    assert (lse - l1).abs().max().item() <= 1e-13


def test_causal_rows_first_and_last():
    """With L = qo_len, new token 0 sees only token 0 (out = its ckv row, exactly); the last new
    token sees the whole request, as a one-token decode with that query does."""
    qo_len = 4
    inp = _small(seed=34, kv_lens=(4, 50), H=2, P=16)
    qn, qp = query_rows(inp, qo_len, seed=35)
    out, lse = oracle.mla_decode_rows(*_rows_args(inp, qn, qp), qo_len, True)
    pg = int(inp.kv_indices[inp.kv_indptr[0]])
    assert torch.equal(out[0], inp.ckv[pg, 0].to(torch.float64).expand_as(out[0]))
    last = torch.tensor([b * qo_len + qo_len - 1 for b in range(inp.batch)])
    o1, l1 = oracle.mla_decode(qn[last], qp[last], inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr,
                               inp.kv_last_page_len, inp.sm_scale)
    assert (out[last] - o1).abs().max().item() <= 1e-13
    assert (lse[last] - l1).abs().max().item() <= 1e-13


def test_non_causal_rows_with_equal_queries_are_equal():
    qo_len = 3
    inp = _small(seed=36, kv_lens=(9, 40), H=2, P=16)
    qn = inp.q_nope.repeat_interleave(qo_len, dim=0)
    qp = inp.q_pe.repeat_interleave(qo_len, dim=0)
    out, lse = oracle.mla_decode_rows(*_rows_args(inp, qn, qp), qo_len, False)
    o1, _ = oracle.mla_decode(*_tiny_args(inp))
    for j in range(qo_len):
        assert (out[j::qo_len] - o1).abs().max().item() <= 1e-13


# ---------------------------------------------------------------- fp16 inputs

def test_f16_decode_all_patterns(lib=None):
    """The oracle's binary16 decoder against torch's float16 -> float64 conversion (a library
    routine) on all 65,536 bit patterns, NaNs included."""
    bits = np.arange(65536, dtype=np.uint16)
    mine = oracle.f16_decode(bits, lib=lib)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    both_nan = np.isnan(mine) & np.isnan(ref)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~both_nan], ref[~both_nan])


@pytest.mark.parametrize("H,P", [(4, 16), (16, 32)])
def test_matches_brute_force_f16(H, P, lib=None):
    """fp16 q, ckv and kpe: the C oracle against the torch fp64 brute force."""
    inp = make_inputs(WORKLOADS["tiny"], kv_lens=[1, 9, 40, 70], batch=4, h_q=H, page_size=P, seed=24, f16=True)
    assert inp.ckv.dtype == torch.float16 and inp.q_nope.dtype == torch.float16
    out, lse = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    ref_out, ref_lse = brute_force(*_tiny_args(inp))
    assert (out - ref_out).abs().max().item() <= 1e-12
    assert (lse - ref_lse).abs().max().item() <= 1e-12


def test_f16_single_token_returns_its_value_row(lib=None):
    inp = make_inputs(WORKLOADS["tiny"], kv_lens=[1], batch=1, h_q=4, page_size=16, seed=25, f16=True)
    out, lse = oracle.mla_decode(*_tiny_args(inp), lib=lib)
    pg = int(inp.kv_indices[0])
    v = inp.ckv[pg, 0].double()
    assert torch.equal(out[0], v.unsqueeze(0).expand(4, 512))
    q = torch.cat([inp.q_nope[0].double(), inp.q_pe[0].double()], dim=1)
    k = torch.cat([v, inp.kpe[pg, 0].double()])
    assert (lse[0] - inp.sm_scale * (q @ k)).abs().max().item() <= 1e-12


# ---------------------------------------------------------------- the pins catch planted mistakes

@pytest.mark.parametrize("plant", [1, 2, 3, 4, 5])
def test_planted_mistakes_are_caught(plant, tmp_path):
    """Copies of the oracle with a dropped kpe term (1), min for max (2), reversed slots (3),
    INT8 codes read unsigned (4), fp16 inputs read as bfloat16 (5): each must fail at least one
    pin above."""
    lib = oracle.load(oracle.build(str(tmp_path / f"liboracle_plant{plant}.so"), plant=plant))
    pins = [lambda: test_golden_closed_form("two_token_ln3.json", lib=lib),
            lambda: test_golden_closed_form("gather_kpe_sign.json", lib=lib),
            lambda: test_matches_brute_force("tiny", lib=lib),
            lambda: test_zero_scale_gives_mean_and_log_length(lib=lib),
            lambda: test_score_shift_moves_only_lse(lib=lib),
            lambda: test_dominant_score_selects_one_row(lib=lib),
            lambda: test_int8_oracle_equals_bf16_oracle_on_exact_codes(lib=lib),
            lambda: test_matches_brute_force_f16(4, 16, lib=lib)]
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"planted mistake {plant} slipped past every pin"
