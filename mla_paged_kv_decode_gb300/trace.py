"""Per-tile timeline of the two-CTA (64/128-head) kernel, for performance work.

    python -m mla_paged_kv_decode_gb300.trace          # from the repository root, on a GPU

Builds a copy of the library with ``-DMLA_TRACE`` (``libmla_decode_trace.so`` beside the normal
one; the kernels then record ``globaltimer`` stamps, 0.256 µs apart, at fixed points), runs the
compute-shaped workload (128 requests × 8192 tokens × 128 heads, page 64) five times untraced
and once traced, and prints the median length of each link of the per-tile chain of the first
cluster: rank 0's K-chunk copies and score MMAs, its softmax and P hand-off, rank 1's values.
The normal library is untouched; nothing here is used by the decode itself.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _binding, build as _build

TRACE_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla_decode_trace.so")


def _median(x: torch.Tensor) -> float:
    x = x[torch.isfinite(x)]
    return float(x.median()) / 1e3 if x.numel() else float("nan")


def pair_chain(workload: str = "compute") -> dict:
    from workloads import WORKLOADS, make_inputs   # the repository's seeded input generators

    import mla_paged_kv_decode_gb300 as mla

    _build.build(out=TRACE_LIB, extra=("-DMLA_TRACE",))
    lib = mla.load(TRACE_LIB)
    _binding._lib = lib
    lib.mla_debug_set_trace.restype = None
    lib.mla_debug_set_trace.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    inp = make_inputs(WORKLOADS[workload])
    assert inp.h_q >= 64 and inp.ckv_scale is None, "the two-CTA kernel serves 64/128 heads over a bf16 cache"
    d = inp.to("cuda")
    dec = mla.Decoder(inp.kv_indptr, inp.kv_last_page_len, inp.h_q, inp.page_size)
    out = torch.empty(inp.batch, inp.h_q, 512, device="cuda")
    lse = torch.empty(inp.batch, inp.h_q, device="cuda")
    nctas = lib.mla_plan_num_ctas(dec.plan.handle)
    # [CTA 0..1][event 0..7][tile 0..255], then CTA 0's per-chunk stamps [lane 0..3][chunk 0..1023]
    # in the area of CTAs 2 and 3, then 8 milestones per CTA
    tr = torch.zeros(4 * 8 * 256 + nctas * 8, dtype=torch.int64, device="cuda")

    def run():
        dec.run(d.q_nope, d.q_pe, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len, inp.sm_scale,
                out=out, lse=lse)

    for _ in range(5):
        run()
    lib.mla_debug_set_trace(dec.plan.handle, ctypes.c_void_p(tr.data_ptr()))
    tr.zero_()
    torch.cuda.synchronize()
    run()
    torch.cuda.synchronize()
    assert dec.device_status() == mla.MLA_OK
    t = tr.cpu().double()
    ev = t[: 2 * 8 * 256].view(2, 8, 256)
    unit = t[2 * 8 * 256: 4 * 8 * 256].view(4, 1024)
    r0, r1 = ev[0], ev[1]
    n = int((r0[1] > 0).sum())
    s = slice(2, n - 1)   # steady state: skip the first tiles and the last
    nk = int((unit[1] > 0).sum())
    acq, iss, land, rel = unit[0, :nk], unit[1, :nk], unit[2, :nk], unit[3, :nk]
    return {
        "tiles (first cluster)": n,
        "period, scores start to scores start": _median(r0[1, 3:n] - r0[1, 2:n - 1]),
        "scores issue, first MMA to last": _median(r0[2, s] - r0[1, s]),
        "K chunk issue interval": _median(iss[1:] - iss[:-1]),
        "producer wait for a free K slot": _median(acq[1:] - iss[:-1]),
        "K chunk issued -> landed": _median(land - iss),
        "K chunk landed -> its MMAs issued": _median(rel - land),
        "softmax: TMEM load": _median(r0[6, s] - r0[3, s]),
        "softmax: softmax and P staging": _median(r0[7, s] - r0[6, s]),
        "softmax: P copy issue": _median(r0[4, s] - r0[7, s]),
        "P staged (rank 0) -> values start (rank 1)": _median(r1[5, s] - r0[7, s]),
        "values issue (rank 1)": _median(r1[6, s] - r1[5, s]),
        "values issued -> P buffer returned": _median(r1[7, s] - r1[6, s]),
    }


if __name__ == "__main__":
    for k, v in pair_chain().items():
        print(f"{k:>45}: {v:8.3f} us" if isinstance(v, float) else f"{k:>45}: {v}")
