"""TEST INFRASTRUCTURE: a second, independent fp64 statement of MLA decode.

It materialises each request's keys K = [ckv | kpe] and values V = ckv by
plain Python indexing over the page list and hands the rest to library
routines (``torch.softmax``, ``torch.logsumexp``, matmul).  It shares nothing
with ``mla_oracle.c`` and exists to pin it on small shapes.  Absorbed MLA as
single-KV-head MQA with qk dim 512 + 64 and v dim 512 follows "Benchmarking
MLA" (FlashInfer issue #700); the paged buffers follow FlashInfer PR #844.
"""
from __future__ import annotations

import torch


def _dequant_e4m3(codes: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    return codes.view(torch.float8_e4m3fn).to(torch.float64) * scale.to(torch.float64).unsqueeze(-1)


def _dequant(ckv: torch.Tensor, scale) -> torch.Tensor:
    """The cache in fp64: bf16 as is; uint8 as e4m3 codes, int8 as integers, times the token's scale."""
    if ckv.dtype == torch.uint8:
        return _dequant_e4m3(ckv, scale)
    if ckv.dtype == torch.int8:
        return ckv.to(torch.float64) * scale.to(torch.float64).unsqueeze(-1)
    return ckv.to(torch.float64)


def brute_force(q_nope, q_pe, ckv, kpe, kv_indices, kv_indptr, kv_last_page_len, sm_scale,
                ckv_scale=None):
    B, H, Dc = q_nope.shape
    P = ckv.shape[1]
    ckv64 = _dequant(ckv, ckv_scale)
    kpe64 = kpe.to(torch.float64)
    out = torch.zeros(B, H, Dc, dtype=torch.float64)
    lse = torch.full((B, H), float("-inf"), dtype=torch.float64)
    indptr = [int(x) for x in kv_indptr]
    for b in range(B):
        pages = [int(x) for x in kv_indices[indptr[b]:indptr[b + 1]]]
        if not pages:
            continue
        L = (len(pages) - 1) * P + int(kv_last_page_len[b])
        rows_c, rows_r = [], []
        for t in range(L):
            pg, sl = pages[t // P], t % P
            rows_c.append(ckv64[pg, sl])
            rows_r.append(kpe64[pg, sl])
        V = torch.stack(rows_c)                        # [L, 512]
        K = torch.cat([V, torch.stack(rows_r)], dim=1)  # [L, 576]
        Q = torch.cat([q_nope[b].to(torch.float64), q_pe[b].to(torch.float64)], dim=1)  # [H, 576]
        S = (Q @ K.T) * sm_scale                       # [H, L]
        out[b] = torch.softmax(S, dim=1) @ V
        lse[b] = torch.logsumexp(S, dim=1)
    return out, lse


def brute_force_rows(q_nope, q_pe, ckv, kpe, kv_indices, kv_indptr, kv_last_page_len, sm_scale, qo_len,
                     causal, ckv_scale=None):
    """Several query tokens per request (row b * qo_len + j is new token j of request b, the new
    tokens being the last qo_len of the cache), written as a mask: the scores of the whole
    request are formed and those of tokens after the row's own position are set to -inf
    before ``torch.softmax``."""
    R, H, Dc = q_nope.shape
    B = R // qo_len
    P = ckv.shape[1]
    ckv64 = _dequant(ckv, ckv_scale)
    kpe64 = kpe.to(torch.float64)
    out = torch.zeros(R, H, Dc, dtype=torch.float64)
    lse = torch.full((R, H), float("-inf"), dtype=torch.float64)
    indptr = [int(x) for x in kv_indptr]
    for b in range(B):
        pages = [int(x) for x in kv_indices[indptr[b]:indptr[b + 1]]]
        if not pages:
            continue
        L = (len(pages) - 1) * P + int(kv_last_page_len[b])
        V = torch.stack([ckv64[pages[t // P], t % P] for t in range(L)])
        K = torch.cat([V, torch.stack([kpe64[pages[t // P], t % P] for t in range(L)])], dim=1)
        pos = torch.arange(L)
        for j in range(qo_len):
            r = b * qo_len + j
            Q = torch.cat([q_nope[r].to(torch.float64), q_pe[r].to(torch.float64)], dim=1)
            S = (Q @ K.T) * sm_scale
            if causal:
                S = S.masked_fill(pos > L - qo_len + j, float("-inf"))
            if not torch.isfinite(S).any():
                continue
            out[r] = torch.softmax(S, dim=1) @ V
            lse[r] = torch.logsumexp(S, dim=1)
    return out, lse
