"""Two variants of the decode through the C ABI, against the fp64 oracle.

* Several new tokens per request (qo_len > 1): row b * qo_len + j is new token j of request
  b; causal, it attends to the first L_b - (qo_len - 1 - j) tokens of the request's cache
  ("perf: MLA decode kernel implemented by CuTe targeted to SM80": its tests carry
  batch_size * qo_len query rows).  Checked against ``oracle.mla_decode_rows`` for every
  kernel and cache kind (16/32 heads, 64/128 heads; bf16, fp16, e4m3 and INT8 caches), with
  requests shorter than qo_len (rows with no token) and requests split over several CTAs.
* bf16 output: the same run with MLA_OUT_BF16 must give, bit for bit, the fp32 result
  rounded to nearest even, and the same lse.
"""
import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
import oracle
from gpu_helpers import assert_parity, kv_dtype_of
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


def _inputs(lens, H, P, seed, cache="bf16"):
    return make_inputs(WORKLOADS["tiny"], kv_lens=list(lens), batch=len(lens), h_q=H, page_size=P, seed=seed,
                       fp8=cache == "fp8", int8=cache == "int8", f16=cache == "f16")


def _run(inp, qn, qp, qo_len=1, causal=True, out_dtype=mla.MLA_OUT_F32, sms=None):
    d = inp.to("cuda")
    kvd = kv_dtype_of(inp)
    dec = mla.Decoder(inp.kv_indptr, inp.kv_last_page_len, inp.h_q, inp.page_size, kv_dtype=kvd, sms=sms,
                      qo_len=qo_len, causal=causal, out_dtype=out_dtype)
    out, lse = dec.run(qn.cuda(), qp.cuda(), d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len,
                       inp.sm_scale, ckv_scale=d.ckv_scale)
    torch.cuda.synchronize()
    word = int(dec.workspace[:4].view(torch.int32).item())
    assert dec.device_status() == mla.MLA_OK, f"device status word {word:#x}"
    return out.cpu(), lse.cpu()


ROW_CASES = [
    # H, P, qo_len, causal, cache
    (16, 16, 2, True, "bf16"),
    (32, 64, 3, False, "bf16"),
    (16, 32, 4, True, "bf16"),
    (64, 32, 2, True, "bf16"),
    (128, 64, 3, True, "bf16"),
    (16, 64, 2, True, "fp8"),
    (64, 16, 2, True, "fp8"),
    (16, 64, 3, True, "int8"),
    (64, 32, 2, False, "int8"),
    (16, 16, 2, True, "f16"),
    (128, 64, 2, True, "f16"),
]


@pytest.mark.parametrize("H,P,qo_len,causal,cache", ROW_CASES)
def test_query_rows(H, P, qo_len, causal, cache):
    lens = [0, 1, 2, 3, 33, 700, 3000]
    inp = _inputs(lens, H, P, seed=60 + H + P + qo_len, cache=cache)
    qn, qp = query_rows(inp, qo_len, seed=61 + qo_len, f16=cache == "f16")
    out, lse = _run(inp, qn, qp, qo_len, causal)
    assert out.shape == (len(lens) * qo_len, H, 512)
    ref = oracle.mla_decode_rows(qn, qp, inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr, inp.kv_last_page_len,
                                 inp.sm_scale, qo_len, causal, ckv_scale=inp.ckv_scale)
    assert_parity(out, lse, *ref)


@pytest.mark.parametrize("H,P,cache", [(16, 64, "bf16"), (32, 16, "bf16"), (64, 64, "bf16"), (128, 32, "bf16"),
                                       (16, 16, "fp8"), (128, 64, "fp8"), (16, 32, "int8"), (128, 16, "int8"),
                                       (32, 64, "f16"), (64, 16, "f16")])
def test_bf16_output_is_the_rounded_fp32_output(H, P, cache):
    lens = [0, 1, 129, 2000, 77, 5000]
    inp = _inputs(lens, H, P, seed=70 + H + P, cache=cache)
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
