"""Parity of the fp16-input path (q_nope, q_pe, ckv and kpe in IEEE fp16) with the fp64 oracle.

FlashMLA PR #233 ("Summary") describes its decode kernel as taking "bf16 / fp16" inputs; here
fp16 inputs run on the same kernels as bf16 ones (the warp-MMA kernel up to 32 heads, the
two-CTA tcgen05 kernel for 64 and 128) with f16 MMAs, P rounded to fp16 instead of bf16.  The
oracle decodes every fp16 value exactly; the bars are the bf16 ones (fp16 carries more mantissa
bits than bf16, so they hold with room).  Cases: ragged lengths over the head counts and page
sizes, split patterns, bit-identical reruns, and the full-size memory- and compute-bound shapes
on sampled requests.
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


def _small_f16(kv_lens, H, P, seed):
    return make_inputs(WORKLOADS["tiny"], kv_lens=list(kv_lens), batch=len(kv_lens), h_q=H, page_size=P, seed=seed,
                       f16=True)


@pytest.mark.parametrize("H", [16, 32, 64, 128])
@pytest.mark.parametrize("P", [16, 32, 64])
def test_f16_small_ragged(H, P):
    lens = [1, 17, P, P + 1, 127, 128, 129, 300, 1000, 2049]
    inp = _small_f16(lens, H, P, seed=80 + H + P)
    assert inp.q_nope.dtype == torch.float16 and inp.ckv.dtype == torch.float16
    out, lse, _, _ = run_gpu(inp)
    assert_parity(out, lse, *oracle.decode_inputs(inp))


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("sms", [1, 3, 152])
def test_f16_split_patterns(H, sms):
    inp = _small_f16([3000, 5, 700, 4096, 129], H, 64, seed=81)
    out, lse, _, _ = run_gpu(inp, sms=sms)
    assert_parity(out, lse, *oracle.decode_inputs(inp))


@pytest.mark.parametrize("H", [16, 128])
def test_f16_reruns_are_bit_identical(H):
    inp = _small_f16([2500, 40, 900], H, 32, seed=82)
    out0, lse0, dec, d = run_gpu(inp)
    for _ in range(3):
        o, l = dec.run(d.q_nope, d.q_pe, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len, inp.sm_scale)
        torch.cuda.synchronize()
        assert torch.equal(o.cpu(), out0) and torch.equal(l.cpu(), lse0)


@pytest.mark.parametrize("name,requests", [("membound", [0, 31, 63]), ("compute", [0, 64, 127])])
def test_f16_full_size_sampled(name, requests):
    inp = make_inputs(WORKLOADS[name], f16=True)
    out, lse, _, _ = run_gpu(inp)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    idx = torch.tensor(requests)
    assert_parity(out[idx], lse[idx], *oracle_subset(inp, requests))
