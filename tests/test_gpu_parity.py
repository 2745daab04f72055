"""Parity of the CUDA path with the fp64 oracle, through the C ABI.

Small cases are compared element by element over the whole output; the
full-size workloads (in the launch configuration bench.py times: the device's
SM count) are compared on sampled requests, all heads and all 512 dims of
each.  Edge cases: empty requests, one-token requests, ragged tails inside a
page and inside a tile, single requests split over every SM, NaN in every
slot and page the method must not read, page-placement permutations
(bit-identical), reruns and CUDA-graph replays (bit-identical), and stream order across
back-to-back launches (each kernel's prologue overlaps the previous kernel's tail).
"""
import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
import oracle
from gpu_helpers import assert_parity, oracle_subset, run_gpu
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_kv_decode_gb300 import build as lib_build
    if lib_build.needs_build():
        lib_build.build()
    mla.load()


def _small(kv_lens, H, P, seed, pool=None):
    return make_inputs(WORKLOADS["tiny"], kv_lens=list(kv_lens), batch=len(kv_lens), h_q=H, page_size=P,
                       pool_pages=pool, seed=seed)


def test_tiny_workload():
    inp = make_inputs(WORKLOADS["tiny"])
    out, lse, _, _ = run_gpu(inp)
    ref = oracle.decode_inputs(inp)
    assert_parity(out, lse, *ref)
    # kv_len = 1: the output is that token's ckv row up to the bf16 rounding of P = 1 (exact)
    pg = int(inp.kv_indices[0])
    assert torch.allclose(out[0], inp.ckv[pg, 0].float().expand_as(out[0]), atol=1e-6)


@pytest.mark.parametrize("H", [16, 32, 64, 128])
@pytest.mark.parametrize("P", [16, 32, 64])
def test_small_ragged(H, P):
    lens = [1, 17, P, P + 1, 127, 128, 129, 300, 1000, 2049]
    inp = _small(lens, H, P, seed=100 + H + P, pool=sum((L + P - 1) // P for L in lens) + 5)
    out, lse, _, _ = run_gpu(inp)
    assert_parity(out, lse, *oracle.decode_inputs(inp))


@pytest.mark.parametrize("sms", [1, 3, 152])
def test_split_patterns(sms):
    """The same batch planned for different CTA counts: pieces and merges differ, parity holds."""
    inp = _small([3000, 5, 700, 4096, 129], 16, 64, seed=7)
    out, lse, _, _ = run_gpu(inp, sms=sms)
    assert_parity(out, lse, *oracle.decode_inputs(inp))


@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("sms", [3, 152])
def test_split_patterns_wide_heads(H, sms):
    """64 and 128 heads on the two-CTA kernel: pieces merged over 64 or 128 heads."""
    inp = _small([3000, 5, 700, 4096, 129], H, 64, seed=13 + H)
    out, lse, _, _ = run_gpu(inp, sms=sms)
    assert_parity(out, lse, *oracle.decode_inputs(inp))


@pytest.mark.parametrize("L", [1, 130, 5000])
def test_single_request_64_heads(L):
    """One 64-head request: the kernel's 128-row query box runs past the query tensor."""
    inp = _small([L], 64, 32, seed=14)
    out, lse, _, _ = run_gpu(inp)
    assert_parity(out, lse, *oracle.decode_inputs(inp))


def test_one_long_request_split_into_many_pieces():
    """A lone 32768-token request: the plan cuts it into a few tens of pieces (it weighs their
    merge against the streaming time), more than 8, so the last piece merges them in several
    rounds of 8."""
    inp = _small([32768], 16, 16, seed=8)
    out, lse, dec, _ = run_gpu(inp)
    assert mla.mla_plan_num_partials(dec.plan) > 16
    assert_parity(out, lse, *oracle.decode_inputs(inp))


def test_empty_requests():
    inp = _small([0, 40, 0, 0, 260, 0], 32, 16, seed=9, pool=30)
    out, lse, _, _ = run_gpu(inp)
    ref_out, ref_lse = oracle.decode_inputs(inp)
    assert torch.isneginf(lse[0]).all() and torch.equal(out[0], torch.zeros_like(out[0]))
    assert_parity(out, lse, ref_out, ref_lse)


def test_nan_padding_is_never_read():
    inp = _small([5, 33, 200], 16, 64, seed=10, pool=12)
    assert torch.isnan(inp.ckv.float()).any() and torch.isnan(inp.kpe.float()).any()
    out, lse, _, _ = run_gpu(inp)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    assert_parity(out, lse, *oracle.decode_inputs(inp))


def test_reruns_and_graph_replay_are_bit_identical():
    inp = _small([4000, 77, 1500, 9000], 64, 64, seed=11)
    out0, lse0, dec, d = run_gpu(inp)
    outs = []
    for _ in range(5):
        o, l = dec.run(d.q_nope, d.q_pe, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len, inp.sm_scale)
        outs.append((o.clone(), l.clone()))
    torch.cuda.synchronize()
    for o, l in outs:
        assert torch.equal(o.cpu(), out0) and torch.equal(l.cpu(), lse0)
    # CUDA graph capture of run(); replay into the captured buffers
    s = torch.cuda.Stream()
    out_g = torch.empty_like(d.q_nope, dtype=torch.float32)
    lse_g = torch.empty(inp.batch, inp.h_q, dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        dec.run(d.q_nope, d.q_pe, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len, inp.sm_scale,
                out=out_g, lse=lse_g, stream=s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            dec.run(d.q_nope, d.q_pe, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len, inp.sm_scale,
                    out=out_g, lse=lse_g, stream=s)
    for _ in range(3):
        out_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g.cpu(), out0) and torch.equal(lse_g.cpu(), lse0)


def test_back_to_back_decodes_keep_stream_order():
    """Every decode is launched with programmatic dependent launch: its prologue may overlap the
    previous kernel's tail, but its reads of the caller's buffers and all its writes follow that
    kernel.  Two different decodes alternate into one output buffer with no synchronisation: the
    buffer must end up holding the last one's result, bit for bit.  A torch kernel that rewrites
    q between two launches must be seen by the second."""
    a = _small([3000, 129, 700, 1], 16, 64, seed=31)
    b = _small([50, 2500, 64, 900], 16, 64, seed=32)
    ref_a, lse_ref_a, dec_a, da = run_gpu(a)
    ref_b, lse_ref_b, dec_b, db = run_gpu(b)
    assert not torch.equal(ref_a, ref_b)
    out = torch.empty(a.batch, a.h_q, 512, device="cuda")
    lse = torch.empty(a.batch, a.h_q, device="cuda")
    args = lambda d, inp: (d.q_nope, d.q_pe, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len,
                           inp.sm_scale)
    for _ in range(20):
        dec_a.run(*args(da, a), out=out, lse=lse)
        dec_b.run(*args(db, b), out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), ref_b) and torch.equal(lse.cpu(), lse_ref_b)
    # q rewritten by a torch kernel between two launches on the same stream
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    dec_b.run(*args(db, b), out=out, lse=lse)
    db.q_nope.neg_()
    dec_b.run(*args(db, b), out=out2, lse=lse2)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), ref_b)
    o3, l3 = dec_b.run(*args(db, b))
    torch.cuda.synchronize()
    assert torch.equal(out2.cpu(), o3.cpu()) and torch.equal(lse2.cpu(), l3.cpu())
    assert not torch.equal(out2.cpu(), ref_b)
    assert dec_a.device_status() == mla.MLA_OK and dec_b.device_status() == mla.MLA_OK


def test_page_permutation_is_bit_identical():
    inp = _small([700, 2000, 129], 32, 32, seed=12, pool=100)
    out0, lse0, _, _ = run_gpu(inp)
    g = torch.Generator().manual_seed(3)
    perm = torch.randperm(inp.num_pages, generator=g)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(inp.num_pages)
    inp.ckv = inp.ckv[perm].contiguous()
    inp.kpe = inp.kpe[perm].contiguous()
    inp.kv_indices = inv[inp.kv_indices.long()].to(torch.int32)
    out1, lse1, _, _ = run_gpu(inp)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


@pytest.mark.parametrize("name,sample", [
    ("membound", [0, 17, 40, 63]),
    ("compute", [0, 64, 127]),
    ("b768_kv1024", [0, 333, 767]),
    ("b768_kv2048", [5, 400, 766]),
    ("ragged", None),
])
def test_full_size_workloads_sampled(name, sample):
    inp = make_inputs(WORKLOADS[name])
    out, lse, _, _ = run_gpu(inp)
    if sample is None:
        # ragged: the longest, the shortest and a few in between
        order = torch.argsort(inp.kv_lens)
        sample = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1]), int(order[-2]), 1})
    ref_out, ref_lse = oracle_subset(inp, sample)
    idx = torch.tensor(sample)
    assert_parity(out[idx], lse[idx], ref_out, ref_lse)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
