"""TEST INFRASTRUCTURE: the fp64 oracle of one MLA decode layer (the absorbed form).

Only ``tests/`` and ``bench.py`` may import it; the product path never does.

FlashMLA PR #233 ("What is added": a fused decode layer -- a prologue kernel for RoPE, the
cache write and quantise-on-write, the projections, and the layer as one CUDA graph;
"Performance": a DeepSeek-V2-Lite-shaped layer at 4096 cached tokens) names the layer's steps
and no more.  The reading taken: the absorbed MLA layer of "Benchmarking MLA" (FlashInfer
issue #700: attention as MQA over the latent, K = ckv ‖ kpe, V = ckv), with the key
up-projection W_UK folded into the query and the value up-projection W_UV applied to the
attention output:

    q        = x W_q,  q_nope = q[..., :D_NOPE],  q_pe = q[..., D_NOPE:]
    q_abs[h] = q_nope[h] W_UK[h]
    c        = x W_kv,   k_pe = x W_kpe
    prologue: q_pe and k_pe rotated at the new token's position, c and the rotated k_pe
              written into the paged cache (quantised for an 8-bit cache)
    o_lat    = attention(q_abs, rotated q_pe; cache)
    o[h]     = o_lat[h] W_UV[h],   y = o W_o   (o's heads side by side)

Every step runs in fp64; every activation the layer stores as a bf16 tensor (q, q_abs, c,
k_pe, the rotated q_pe and k_pe, o_lat, o, y) is rounded to bf16 here too.  The attention is
``oracle.mla_decode`` and the prologue ``oracle.decode_prologue``, both pinned on their own.
``plant`` (tests only) makes one deliberate mistake, to show that the layer's pins catch it.
"""
from __future__ import annotations

import torch

from . import decode_prologue, mla_decode

PLANTS = ("skip_cache_write", "swap_uk_heads", "swap_uv_heads", "o_head_order", "q_pe_unrotated")


def _bf(t: torch.Tensor) -> torch.Tensor:
    """fp64 -> bf16 (round to nearest even) -> fp64."""
    return t.to(torch.bfloat16).to(torch.float64)


def decode_layer(x, w, ckv_cache, kpe_cache, kv_indices, kv_indptr, kv_last_page_len, rope_cos_sin, sm_scale,
                 interleaved: bool = False, ckv_scale=None, plant: str = ""):
    """One decode step of one layer on CPU tensors.

    x [B, D] bf16 (the new tokens' hidden states; token b is the last of request b's cache);
    ``w`` has bf16 w_q [D, H, dn + 64], w_kv [D, 512], w_kpe [D, 64], w_uk [H, dn, 512],
    w_uv [H, 512, dv], w_o [H * dv, D].  Returns (y [B, D] as fp64 holding bf16 values, and the
    caches after the prologue: ckv, kpe, scale)."""
    assert plant in ("",) + PLANTS, plant
    B = x.shape[0]
    H, dn, _ = w.w_uk.shape
    f = lambda t: t.to(torch.float64)
    xf = f(x)
    q = _bf(xf @ f(w.w_q).reshape(xf.shape[1], -1)).reshape(B, H, -1)
    q_nope, q_pe = q[:, :, :dn], q[:, :, dn:]
    w_uk = f(w.w_uk)
    if plant == "swap_uk_heads":
        w_uk = torch.roll(w_uk, 1, dims=0)
    q_abs = _bf(torch.einsum("bhd,hde->bhe", q_nope, w_uk))
    c = _bf(xf @ f(w.w_kv))
    k_pe = _bf(xf @ f(w.w_kpe))
    bf = torch.bfloat16
    q_rot, ckv2, kpe2, sc2 = decode_prologue(q_pe.to(bf), c.to(bf), k_pe.to(bf), rope_cos_sin, kv_indices, kv_indptr,
                                             kv_last_page_len, 1, interleaved, ckv_cache, kpe_cache, ckv_scale)
    if plant == "skip_cache_write":
        ckv2, kpe2, sc2 = ckv_cache, kpe_cache, ckv_scale
    if plant == "q_pe_unrotated":
        q_rot = q_pe.to(bf)
    o_lat, _ = mla_decode(q_abs.to(bf), q_rot, ckv2, kpe2, kv_indices, kv_indptr, kv_last_page_len, sm_scale,
                          ckv_scale=sc2)
    o_lat = _bf(o_lat)
    w_uv = f(w.w_uv)
    if plant == "swap_uv_heads":
        w_uv = torch.roll(w_uv, 1, dims=0)
    o = _bf(torch.einsum("bhe,hev->bhv", o_lat, w_uv))
    o_flat = o.transpose(1, 2).reshape(B, -1) if plant == "o_head_order" else o.reshape(B, -1)
    y = _bf(o_flat @ f(w.w_o))
    return y, ckv2, kpe2, sc2
