"""The decode prologue kernel (RoPE, cache write, quantise-on-write) through the C ABI, against
the oracle's ``decode_prologue``, then a decode over the updated cache against the oracle, for
the bf16, e4m3, INT8 and fp16 caches.

The latent written to the cache (16-bit bits, or 8-bit codes and fp32 scales) must be identical;
the rotated q_pe and kpe are fp32 rotations rounded to the 16-bit type on one side and fp64 ones
on the other, so they may differ by one unit in the last place; every entry the prologue does not
own keeps its bits (NaN padding included)."""
import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
import oracle
from gpu_helpers import assert_parity
from workloads import WORKLOADS, make_inputs, new_tokens, rope_table

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_kv_decode_gb300 import build as lib_build
    if lib_build.needs_build():
        lib_build.build()
    mla.load()


def _close16(a, b):
    """Equal bits, or both finite and within one unit in the last place of their 16-bit type
    (bf16: 2^-7 relative, fp16: 2^-10)."""
    a, b = a.cpu(), b.cpu()
    same = a.view(torch.int16) == b.view(torch.int16)
    af, bf = a.float(), b.float()
    ulp = 2.0 ** -10 if a.dtype == torch.float16 else 2.0 ** -7
    near = torch.isfinite(af) & torch.isfinite(bf) & ((af - bf).abs() <= bf.abs() * ulp)
    return bool((same | near).all())


CASES = [
    # H, P, qo_len, cache, interleaved
    (16, 64, 1, "bf16", True),
    (128, 16, 2, "bf16", False),
    (16, 32, 2, "e4m3", True),
    (64, 64, 1, "e4m3", False),
    (16, 64, 2, "int8", False),
    (128, 32, 1, "int8", True),
    (16, 16, 2, "f16", True),
    (128, 64, 1, "f16", False),
]


@pytest.mark.parametrize("H,P,qo_len,cache,interleaved", CASES)
def test_prologue_then_decode(H, P, qo_len, cache, interleaved):
    lens = [1, 2, 17, 300, 2500]
    fp8, f16 = cache == "e4m3", cache == "f16"
    inp = make_inputs(WORKLOADS["tiny"], kv_lens=lens, batch=len(lens), h_q=H, page_size=P, seed=100 + H + P,
                      fp8=fp8, int8=cache == "int8", f16=f16)
    q_pe, ckv_new, kpe_new = new_tokens(inp, qo_len, seed=101, f16=f16)
    table = rope_table(max(lens) + 1)
    rq, rckv, rkpe, rsc = oracle.decode_prologue(q_pe, ckv_new, kpe_new, table, inp.kv_indices, inp.kv_indptr,
                                                 inp.kv_last_page_len, qo_len, interleaved, inp.ckv, inp.kpe,
                                                 ckv_scale=inp.ckv_scale)
    d = inp.to("cuda")
    # rows the prologue leaves untouched keep the input; the interleaved cases rotate in place
    q_in = q_pe.cuda()
    q_out = q_in if interleaved else q_in.clone()
    kvd = {"bf16": mla.MLA_KV_BF16, "e4m3": mla.MLA_KV_FP8_E4M3, "int8": mla.MLA_KV_INT8, "f16": mla.MLA_KV_F16}[cache]
    eight = cache in ("e4m3", "int8")
    mla.mla_decode_prologue(inp.batch, qo_len, H, P, kvd, interleaved, q_in, q_out, ckv_new.cuda(),
                            kpe_new.cuda(), table.cuda(), d.kv_indices, d.kv_indptr, d.kv_last_page_len, d.ckv,
                            d.ckv_scale, d.kpe)
    torch.cuda.synchronize()
    gckv = d.ckv.cpu()
    if eight:
        assert torch.equal(gckv, rckv)
        assert torch.equal(d.ckv_scale.cpu().view(torch.int32), rsc.view(torch.int32))
    else:
        assert torch.equal(gckv.view(torch.int16), rckv.view(torch.int16))
    assert _close16(d.kpe, rkpe)
    assert _close16(q_out, rq)

    # decode over the updated cache: query rows [q_nope | rotated q_pe]
    qn = torch.randn(inp.batch * qo_len, H, 512, generator=torch.Generator().manual_seed(102)).to(
        torch.float16 if f16 else torch.bfloat16)
    dec = mla.Decoder(inp.kv_indptr, inp.kv_last_page_len, H, P, kv_dtype=kvd, qo_len=qo_len, causal=True)
    out, lse = dec.run(qn.cuda(), q_out, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len, inp.sm_scale,
                       ckv_scale=d.ckv_scale)
    torch.cuda.synchronize()
    assert dec.device_status() == mla.MLA_OK
    ref = oracle.mla_decode_rows(qn, q_out.cpu(), gckv, d.kpe.cpu(), inp.kv_indices, inp.kv_indptr,
                                 inp.kv_last_page_len, inp.sm_scale, qo_len, True,
                                 ckv_scale=d.ckv_scale.cpu() if eight else None)
    assert_parity(out.cpu(), lse.cpu(), *ref)


def test_prologue_argument_checks():
    inp = make_inputs(WORKLOADS["tiny"], kv_lens=[5], batch=1, h_q=16, page_size=16, seed=103)
    d = inp.to("cuda")
    q_pe, ckv_new, kpe_new = (t.cuda() for t in new_tokens(inp, 1, seed=104))
    table = rope_table(8).cuda()
    with pytest.raises(mla.MLAError):   # an 8-bit cache needs its scales
        mla.mla_decode_prologue(1, 1, 16, 16, mla.MLA_KV_FP8_E4M3, True, q_pe, q_pe, ckv_new, kpe_new, table,
                                d.kv_indices, d.kv_indptr, d.kv_last_page_len, d.ckv, None, d.kpe)
    with pytest.raises(mla.MLAError):   # page size outside the supported set
        mla.mla_decode_prologue(1, 1, 16, 24, mla.MLA_KV_BF16, True, q_pe, q_pe, ckv_new, kpe_new, table,
                                d.kv_indices, d.kv_indptr, d.kv_last_page_len, d.ckv, None, d.kpe)
