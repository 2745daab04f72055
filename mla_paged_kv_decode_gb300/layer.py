"""One MLA decode layer (the absorbed form) around the library's prologue and decode, replayable
as one CUDA graph.

FlashMLA PR #233 ("What is added", "Performance") builds a fused decode layer of a
DeepSeek-V2-Lite-shaped model -- one prologue kernel (RoPE, concat, cache write,
quantise-on-write), the projections, and the whole layer captured as one CUDA graph -- and
times it per layer at 4096 cached tokens.  This module is that layer over this library, with
the projections as plain cuBLAS GEMMs (torch.matmul / bmm) on synthetic weights:

    q        = x W_q                         [B, H, 192]: q_nope (128), q_pe (64, before RoPE)
    q_abs[h] = q_nope[h] W_UK[h]             [B, H, 512]   (the key up-projection, absorbed)
    c        = x W_kv                        [B, 512]      (the new token's latent)
    k_pe     = x W_kpe                       [B, 64]       (before RoPE)
    prologue: RoPE on q_pe and k_pe; c and RoPE(k_pe) written into the paged cache
    o_lat    = decode(q_abs, RoPE(q_pe), cache)             [B, H, 512]
    o[h]     = o_lat[h] W_UV[h]              [B, H, 128]   (the value up-projection)
    y        = o W_o                         [B, 2048]

Every activation is a bf16 tensor (the decode returns its output rounded to bf16); the
new token is the last token of each request's cache.  The caller owns the weights, the
caches and the page table; the plan is built once for the batch's cache lengths.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from ._binding import (MLA_KV_BF16, MLA_OUT_BF16, mla_decode_plan_commit, mla_decode_plan_ex,
                       mla_decode_prologue, mla_decode_run)

# DeepSeek-V2-Lite's shape (the pages give only h_q = 16); the layer takes its sizes from the weights
D_MODEL, N_HEADS, D_NOPE, D_ROPE, D_LATENT, D_V = 2048, 16, 128, 64, 512, 128


@dataclass
class LayerWeights:
    """bf16 weights of one layer: w_q [D, H, dn + 64], w_kv [D, 512], w_kpe [D, 64],
    w_uk [H, dn, 512], w_uv [H, 512, dv], w_o [H * dv, D] (V2-Lite: D 2048, H 16, dn = dv = 128)."""
    w_q: torch.Tensor
    w_kv: torch.Tensor
    w_kpe: torch.Tensor
    w_uk: torch.Tensor
    w_uv: torch.Tensor
    w_o: torch.Tensor

    def to(self, device) -> "LayerWeights":
        return LayerWeights(*(t.to(device).contiguous() for t in (self.w_q, self.w_kv, self.w_kpe, self.w_uk,
                                                                  self.w_uv, self.w_o)))


class DecodeLayer:
    """One decode step of one layer for a fixed batch composition (the cache lengths, which
    include the new token).  ``step`` runs it eagerly; ``capture`` records it as one CUDA graph
    over static buffers, replayed by ``replay``."""

    def __init__(self, weights: LayerWeights, kv_indptr: torch.Tensor, kv_last_page_len: torch.Tensor,
                 page_size: int, rope_cos_sin: torch.Tensor, kv_dtype: int = MLA_KV_BF16,
                 rope_interleaved: bool = False, sm_scale: Optional[float] = None, sms: Optional[int] = None,
                 device=None):
        device = torch.device(device or "cuda")
        self.w = weights
        self.heads, self.d_nope, _ = weights.w_uk.shape
        self.d_v = weights.w_uv.shape[2]
        self.d_model = weights.w_q.shape[0]
        self.batch = int(kv_indptr.numel()) - 1
        self.page_size, self.kv_dtype, self.interleaved = page_size, kv_dtype, rope_interleaved
        # the non-absorbed form's qk head dim (dn + 64) sets the default scale
        self.sm_scale = (self.d_nope + D_ROPE) ** -0.5 if sm_scale is None else sm_scale
        self.rope = rope_cos_sin.to(device=device, dtype=torch.float32).contiguous()
        if sms is None:
            sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.plan = mla_decode_plan_ex(kv_indptr.cpu(), kv_last_page_len.cpu(), self.batch, 1, True, self.heads,
                                       page_size, sms, kv_dtype, MLA_OUT_BF16)
        self.workspace = torch.empty(max(self.plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
        mla_decode_plan_commit(self.plan, self.workspace)
        B, H, bf = self.batch, self.heads, torch.bfloat16
        self.q_pe_rot = torch.empty(B, H, D_ROPE, dtype=bf, device=device)
        self.o_lat = torch.empty(B, H, D_LATENT, dtype=bf, device=device)
        self.lse = torch.empty(B, H, dtype=torch.float32, device=device)
        self.graph = None
        self.static = None

    def step(self, x, ckv_cache, kpe_cache, kv_indices, kv_indptr, kv_last_page_len, ckv_scale=None, stream=None):
        """y [B, 2048] bf16 for the new tokens' hidden states x [B, 2048] bf16; writes the new
        tokens into the caches."""
        B, H, dn = self.batch, self.heads, self.d_nope
        q = torch.matmul(x, self.w.w_q.view(self.d_model, -1)).view(B, H, dn + D_ROPE)
        q_pe = q[:, :, dn:].contiguous()
        q_abs = torch.bmm(q[:, :, :dn].transpose(0, 1), self.w.w_uk).transpose(0, 1).contiguous()
        c_new = torch.matmul(x, self.w.w_kv)
        k_pe = torch.matmul(x, self.w.w_kpe)
        mla_decode_prologue(B, 1, H, self.page_size, self.kv_dtype, self.interleaved, q_pe, self.q_pe_rot,
                            c_new, k_pe, self.rope, kv_indices, kv_indptr, kv_last_page_len, ckv_cache, ckv_scale,
                            kpe_cache, stream)
        mla_decode_run(self.plan, q_abs, self.q_pe_rot, ckv_cache, ckv_scale, kpe_cache, kv_indices, kv_indptr,
                       kv_last_page_len, self.sm_scale, self.o_lat, self.lse, self.workspace, stream)
        o = torch.bmm(self.o_lat.transpose(0, 1), self.w.w_uv).transpose(0, 1).reshape(B, H * self.d_v)
        return torch.matmul(o, self.w.w_o)

    def capture(self, x, ckv_cache, kpe_cache, kv_indices, kv_indptr, kv_last_page_len, ckv_scale=None):
        """Record one step over these (static) buffers as a CUDA graph; returns the graph's output
        buffer.  Refill x (and the caches) in place between replays."""
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):   # warm-up outside the capture (cuBLAS workspaces, handles)
            self.step(x, ckv_cache, kpe_cache, kv_indices, kv_indptr, kv_last_page_len, ckv_scale, stream=stream)
        stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            y = self.step(x, ckv_cache, kpe_cache, kv_indices, kv_indptr, kv_last_page_len, ckv_scale, stream=stream)
        self.static = y
        return y

    def replay(self):
        self.graph.replay()
        return self.static
