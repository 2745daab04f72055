"""Parity of the INT8 cache path (two's-complement codes with one fp32 scale per token, bf16 kpe)
with the fp64 oracle.

FlashMLA PR #233 ("What is added") lists an 8-bit cache "FP8 e4m3 or INT8 with one scale per
token", 644 bytes a token; its "Correctness" section reports the INT8 cache's worst cosine
distance to bf16 as 2.6e-4.  Two references, as for the e4m3 cache:

* the oracle on the dequantised cache (scale_t * code_t), held to the bf16 tolerances: this
  checks the kernel's arithmetic;
* the oracle on the bf16 cache the codes were quantised from, cosine distance <= 3e-3 (the
  8-bit bar): this checks the quantisation end to end.

Cases: ragged lengths over page sizes 16/32/64 and 16/32/64/128 heads, splits over 1, 3 and
every SM, bit-identical reruns, tokens whose magnitudes span six orders (the per-token scales
must stay within the kernel's f16 weights), code -128 with a NaN scale in every unused slot, and
the full-size 8-bit workload shape on sampled requests.
"""
import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
import oracle
from gpu_helpers import COS_DIST_FP8, assert_parity, cos_dist, oracle_subset, run_gpu
from workloads import WORKLOADS, make_inputs, quantize_int8_per_token

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_kv_decode_gb300 import build as lib_build
    if lib_build.needs_build():
        lib_build.build()
    mla.load()


def _small_int8(kv_lens, H, P, seed, pool=None):
    return make_inputs(WORKLOADS["tiny"], kv_lens=list(kv_lens), batch=len(kv_lens), h_q=H, page_size=P,
                       pool_pages=pool, seed=seed, int8=True)


def _check_both(inp, out, lse, requests=None):
    if requests is None:
        ref = oracle.decode_inputs(inp)
        ref16 = oracle.decode_inputs(inp, use_bf16_cache=True)
        o, l = out, lse
    else:
        ref = oracle_subset(inp, requests)
        ref16 = oracle_subset(inp, requests, use_bf16_cache=True)
        idx = torch.tensor(requests)
        o, l = out[idx], lse[idx]
    assert_parity(o, l, *ref)
    cd = cos_dist(o.double(), ref16[0])
    assert cd <= COS_DIST_FP8, f"cosine distance to the bf16-cache oracle {cd:.3e}"
    return cd


@pytest.mark.parametrize("H", [16, 32])
@pytest.mark.parametrize("P", [16, 32, 64])
def test_int8_small_ragged(H, P):
    lens = [1, 17, P, P + 1, 127, 128, 129, 300, 1000, 2049]
    inp = _small_int8(lens, H, P, seed=60 + H + P)
    assert inp.ckv.dtype == torch.int8 and inp.ckv_scale is not None
    out, lse, dec, _ = run_gpu(inp)
    assert mla.mla_plan_heads_per_cta(dec.plan) == H
    _check_both(inp, out, lse)


@pytest.mark.parametrize("H", [64, 128])
def test_int8_wide_heads(H):
    """64 and 128 heads: 32-head CTAs, h_q / 32 of them per unit."""
    inp = _small_int8([1, 100, 129, 700, 2049], H, 64, seed=70 + H)
    out, lse, dec, _ = run_gpu(inp)
    assert mla.mla_plan_heads_per_cta(dec.plan) == 32
    _check_both(inp, out, lse)


@pytest.mark.parametrize("sms", [1, 3, 152])
def test_int8_split_patterns(sms):
    inp = _small_int8([3000, 5, 700, 4096, 129], 16, 64, seed=71)
    out, lse, _, _ = run_gpu(inp, sms=sms)
    _check_both(inp, out, lse)


def test_int8_reruns_are_bit_identical():
    inp = _small_int8([2500, 40, 900], 32, 32, seed=72)
    out0, lse0, dec, d = run_gpu(inp)
    for _ in range(3):
        o, l = dec.run(d.q_nope, d.q_pe, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len, inp.sm_scale,
                       ckv_scale=d.ckv_scale)
        torch.cuda.synchronize()
        assert torch.equal(o.cpu(), out0) and torch.equal(l.cpu(), lse0)


def test_int8_scale_extremes():
    """Tokens scaled by 1e-3 .. 1e3 before quantisation: the running scale maximum moves across
    tiles and the f16 weights p_t s_t / c span both ends."""
    inp = _small_int8([1500, 700], 16, 64, seed=73)
    g = torch.Generator().manual_seed(6)
    fin = torch.nan_to_num(inp.ckv_bf16.float(), nan=0.0)
    mag = 10.0 ** (torch.randint(-3, 4, (fin.shape[0], fin.shape[1], 1), generator=g).float())
    scaled = (fin * mag).to(torch.bfloat16)
    codes, scale = quantize_int8_per_token(scaled)
    bad = ~torch.isfinite(inp.ckv_scale)
    codes[bad] = -128
    scale[bad] = float("nan")
    inp.ckv_bf16 = scaled
    inp.ckv = codes
    inp.ckv_scale = scale
    out, lse, _, _ = run_gpu(inp)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    ref_out, ref_lse = oracle.decode_inputs(inp)
    # scores reach ~1e4 here: bf16 tolerances relative to each request's largest output and |lse|
    for b in range(inp.batch):
        o = out[b].double()
        scale_b = max(1.0, float(ref_out[b].abs().max()))
        err = float((o - ref_out[b]).abs().max())
        assert err <= 2e-2 * scale_b, (b, err, scale_b)
        assert cos_dist(o, ref_out[b]) <= 1e-4
        lerr = float((lse[b].double() - ref_lse[b]).abs().max())
        assert lerr <= 1e-3 + 2e-6 * float(ref_lse[b].abs().max()), (b, lerr)


def test_int8_full_size_sampled():
    inp = make_inputs(WORKLOADS["fp8"], fp8=False, int8=True)
    out, lse, _, _ = run_gpu(inp)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    cd = _check_both(inp, out, lse, requests=[0, 31, 63])
    print(f"INT8 full size: cosine distance to the bf16-cache oracle {cd:.2e}")
