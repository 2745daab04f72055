"""Shared helpers of the GPU tests: run the CUDA path through the C ABI and
compare with the fp64 oracle using the parity gates of the method."""
from __future__ import annotations

import torch

import mla_paged_kv_decode_gb300 as mla
import oracle

# parity gates (bf16 cache): max |out - oracle|, cosine distance of the whole out
# tensor, max |lse - oracle|; the 8-bit cache is held to a cosine distance
# against the oracle on the bf16 cache it was quantised from
MAX_ABS = 2e-2
COS_DIST = 1e-4
LSE_ABS = 1e-3
COS_DIST_FP8 = 3e-3


def cos_dist(a: torch.Tensor, b: torch.Tensor) -> float:
    a = a.double().flatten()
    b = b.double().flatten()
    return float(1.0 - (a @ b) / (a.norm() * b.norm()))


def kv_dtype_of(inp):
    """The cache type of a workloads.Inputs: bf16, e4m3 codes (uint8) or INT8 codes (int8)."""
    if inp.ckv_scale is None:
        return mla.MLA_KV_F16 if inp.ckv.dtype == torch.float16 else mla.MLA_KV_BF16
    return mla.MLA_KV_INT8 if inp.ckv.dtype == torch.int8 else mla.MLA_KV_FP8_E4M3


def run_gpu(inp, sms=None, stream=None):
    """Plan + commit + run on cuda:0; returns (out, lse) on the CPU and the decoder."""
    d = inp.to("cuda")
    kvd = kv_dtype_of(inp)
    dec = mla.Decoder(inp.kv_indptr, inp.kv_last_page_len, inp.h_q, inp.page_size, kv_dtype=kvd, sms=sms,
                      stream=stream)
    out, lse = dec.run(d.q_nope, d.q_pe, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len,
                       inp.sm_scale, ckv_scale=d.ckv_scale, stream=stream)
    torch.cuda.synchronize()
    word = int(dec.workspace[:4].view(torch.int32).item())   # status word: 0x100 | site of a timed-out wait
    assert dec.device_status() == mla.MLA_OK, f"device status word {word:#x}"
    return out.cpu(), lse.cpu(), dec, d


def assert_parity(out, lse, ref_out, ref_lse, max_abs=MAX_ABS, cos=COS_DIST, lse_abs=LSE_ABS, rows=None):
    out = out.double()
    lse = lse.double()
    assert torch.isfinite(out).all(), "non-finite output"
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isfinite(lse), fin), "empty-request lse must be -inf exactly where the oracle's is"
    err = (out - ref_out).abs().max().item()
    cd = cos_dist(out, ref_out) if ref_out.abs().max() > 0 else 0.0
    lerr = (lse[fin] - ref_lse[fin]).abs().max().item() if fin.any() else 0.0
    msg = f"max|out-oracle|={err:.3e} cos_dist={cd:.3e} max|lse-oracle|={lerr:.3e}"
    assert err <= max_abs and cd <= cos and lerr <= lse_abs, msg
    return err, cd, lerr


def oracle_subset(inp, requests, threads=0, use_bf16_cache=False):
    """Oracle on a subset of requests (same cache, sliced q and page lists)."""
    return oracle.decode_subset(inp, requests, threads=threads, use_bf16_cache=use_bf16_cache)
