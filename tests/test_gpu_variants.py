"""Two variants of the decode through the C ABI, against the fp64 oracle.

* Several new tokens per request (qo_len > 1): row b * qo_len + j is new token j of request
  b; causal, it attends to the first L_b - (qo_len - 1 - j) tokens of the request's cache
  ("perf: MLA decode kernel implemented by CuTe targeted to SM80": its tests carry
  batch_size * qo_len query rows).  Checked against ``oracle.mla_decode_rows`` for every
  kernel (16/32 heads, 64/128 heads, the 8-bit cache), with requests shorter than qo_len (rows
  with no token) and requests split over several CTAs.
* bf16 output: the same run with MLA_OUT_BF16 must give, bit for bit, the fp32 result
  rounded to nearest even, and the same lse.
"""
import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
import oracle
from gpu_helpers import assert_parity
from workloads import WORKLOADS, make_inputs, query_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_kv_decode_gb300 import build as lib_build
    if lib_build.needs_build():
        lib_build.build()
    mla.load()


def _inputs(lens, H, P, seed, fp8=False):
    return make_inputs(WORKLOADS["tiny"], kv_lens=list(lens), batch=len(lens), h_q=H, page_size=P, seed=seed,
                       fp8=fp8)


def _run(inp, qn, qp, qo_len=1, causal=True, out_dtype=mla.MLA_OUT_F32, sms=None):
    d = inp.to("cuda")
    kvd = mla.MLA_KV_FP8_E4M3 if inp.ckv_scale is not None else mla.MLA_KV_BF16
    dec = mla.Decoder(inp.kv_indptr, inp.kv_last_page_len, inp.h_q, inp.page_size, kv_dtype=kvd, sms=sms,
                      qo_len=qo_len, causal=causal, out_dtype=out_dtype)
    out, lse = dec.run(qn.cuda(), qp.cuda(), d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len,
                       inp.sm_scale, ckv_scale=d.ckv_scale)
    torch.cuda.synchronize()
    word = int(dec.workspace[:4].view(torch.int32).item())
    assert dec.device_status() == mla.MLA_OK, f"device status word {word:#x}"
    return out.cpu(), lse.cpu()


ROW_CASES = [
    # H, P, qo_len, causal, fp8
    (16, 16, 2, True, False),
    (32, 64, 3, False, False),
    (16, 32, 4, True, False),
    (64, 32, 2, True, False),
    (128, 64, 3, True, False),
    (16, 64, 2, True, True),
    (64, 16, 2, True, True),
]


@pytest.mark.parametrize("H,P,qo_len,causal,fp8", ROW_CASES)
def test_query_rows(H, P, qo_len, causal, fp8):
    lens = [0, 1, 2, 3, 33, 700, 3000]
    inp = _inputs(lens, H, P, seed=60 + H + P + qo_len, fp8=fp8)
    qn, qp = query_rows(inp, qo_len, seed=61 + qo_len)
    out, lse = _run(inp, qn, qp, qo_len, causal)
    assert out.shape == (len(lens) * qo_len, H, 512)
    ref = oracle.mla_decode_rows(qn, qp, inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr, inp.kv_last_page_len,
                                 inp.sm_scale, qo_len, causal, ckv_scale=inp.ckv_scale)
    assert_parity(out, lse, *ref)


@pytest.mark.parametrize("H,P,fp8", [(16, 64, False), (32, 16, False), (64, 64, False), (128, 32, False),
                                     (16, 16, True), (128, 64, True)])
def test_bf16_output_is_the_rounded_fp32_output(H, P, fp8):
    lens = [0, 1, 129, 2000, 77, 5000]
    inp = _inputs(lens, H, P, seed=70 + H + P, fp8=fp8)
    o32, l32 = _run(inp, inp.q_nope, inp.q_pe)
    o16, l16 = _run(inp, inp.q_nope, inp.q_pe, out_dtype=mla.MLA_OUT_BF16)
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(l16, l32)


def test_bf16_output_with_query_rows():
    inp = _inputs([5, 300, 4000, 1], 16, 64, seed=80)
    qn, qp = query_rows(inp, 2, seed=81)
    o32, l32 = _run(inp, qn, qp, 2, True)
    o16, l16 = _run(inp, qn, qp, 2, True, out_dtype=mla.MLA_OUT_BF16)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(l16, l32)
