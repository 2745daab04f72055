"""Seeded synthetic inputs for MLA paged-KV decode.

This module only *draws* inputs: it holds none of the attention arithmetic, so
both the fp64 oracle and the CUDA path can consume what it produces without
sharing any computation.  Shapes follow the absorbed-MLA decode problem as
stated in "perf: MLA decode kernel implemented by CuTe targeted to SM80"
(FlashInfer PR #844, the benchmark's q_nope/q_pe/ckv/kpe buffers and the
gaussian test initialisation) and the paged layout addressed by kv_indptr /
kv_indices / kv_last_page_len.

Recipe (the same for every workload):
  * a torch CPU ``Generator`` seeded with the workload's seed;
  * draw order: request lengths (ragged workloads only), the page
    permutation of the pool (``randperm``), then q_nope, q_pe, ckv, kpe as
    fp32 ``randn`` rounded to bf16;
  * request b's logical pages take the next n_b entries of the permutation,
    so physical placement is scattered;
  * slots past kv_last_page_len on a request's last page, and pool pages no
    request references, are filled with NaN (bf16 NaN; for the 8-bit cache
    code 0x7F and a NaN scale), so any read of them poisons the result;
  * 8-bit cache: per token scale = fp32(absmax over the 512 ckv values) / 448,
    codes = round-to-nearest-even e4m3 of clamp(x / scale, -448, 448), done
    with torch's float8_e4m3fn cast (a library routine); absmax 0 gives scale
    0 and all-zero codes.  kpe stays bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

D_CKV = 512
D_KPE = 64
E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    batch: int
    h_q: int
    page_size: int
    kv_lens: Optional[tuple] = None      # explicit lengths
    kv_len: Optional[int] = None         # uniform length
    ragged_max: Optional[int] = None     # log-uniform lengths in [1, ragged_max]
    pool_pages: Optional[int] = None     # pool size (default: exactly the pages used)
    fp8: bool = False
    sm_scale: float = 1.0 / math.sqrt(192.0)
    description: str = ""


WORKLOADS = {
    "tiny": Workload(
        "tiny", seed=0, batch=4, h_q=16, page_size=16, kv_lens=(1, 17, 64, 203), pool_pages=40,
        description="batch 4, h_q 16, page 16, kv_lens [1,17,64,203], 40-page pool"),
    "membound": Workload(
        "membound", seed=1, batch=64, h_q=16, page_size=64, kv_len=4096,
        description="DeepSeek-V2-Lite-shaped: batch 64, h_q 16, page 64, kv_len 4096"),
    "compute": Workload(
        "compute", seed=2, batch=128, h_q=128, page_size=64, kv_len=8192,
        description="DeepSeek-V3-shaped: batch 128, h_q 128, page 64, kv_len 8192"),
    "b768_kv1024": Workload(
        "b768_kv1024", seed=2, batch=768, h_q=64, page_size=64, kv_len=1024,
        description="batch 768, h_q 64, page 64, kv_len 1024"),
    "b768_kv2048": Workload(
        "b768_kv2048", seed=2, batch=768, h_q=64, page_size=64, kv_len=2048,
        description="batch 768, h_q 64, page 64, kv_len 2048"),
    "ragged": Workload(
        "ragged", seed=3, batch=256, h_q=128, page_size=16, ragged_max=32768,
        description="batch 256, h_q 128, page 16, kv_len log-uniform in [1, 32768]"),
    "fp8": Workload(
        "fp8", seed=4, batch=64, h_q=16, page_size=64, kv_len=16384, fp8=True,
        description="batch 64, h_q 16, page 64, kv_len 16384, e4m3 ckv + fp32 per-token scale"),
}


@dataclass
class Inputs:
    """One batch of decode inputs, all on one device (CPU unless moved)."""
    workload: Workload
    q_nope: torch.Tensor            # bf16 [B, H, 512]
    q_pe: torch.Tensor              # bf16 [B, H, 64]
    ckv: torch.Tensor               # bf16 [num_pages, P, 512]  (fp8: uint8 codes)
    kpe: torch.Tensor               # bf16 [num_pages, P, 64]
    kv_indptr: torch.Tensor         # int32 [B+1]
    kv_indices: torch.Tensor        # int32 [total pages referenced]
    kv_last_page_len: torch.Tensor  # int32 [B]
    kv_lens: torch.Tensor           # int64 [B]  (derived, for convenience)
    ckv_scale: Optional[torch.Tensor] = None  # fp32 [num_pages, P] for the 8-bit cache
    ckv_bf16: Optional[torch.Tensor] = None   # the bf16 cache the 8-bit one was quantised from
    extra: dict = field(default_factory=dict)

    @property
    def batch(self):
        return self.q_nope.shape[0]

    @property
    def h_q(self):
        return self.q_nope.shape[1]

    @property
    def page_size(self):
        return self.ckv.shape[1]

    @property
    def num_pages(self):
        return self.ckv.shape[0]

    @property
    def sm_scale(self):
        return self.workload.sm_scale

    def to(self, device) -> "Inputs":
        mv = lambda t: None if t is None else t.to(device)
        return Inputs(self.workload, mv(self.q_nope), mv(self.q_pe), mv(self.ckv), mv(self.kpe),
                      mv(self.kv_indptr), mv(self.kv_indices), mv(self.kv_last_page_len),
                      self.kv_lens.clone(), mv(self.ckv_scale), mv(self.ckv_bf16), dict(self.extra))


def ragged_lengths(gen: torch.Generator, batch: int, max_len: int) -> list:
    """kv_len = clamp(round(exp(u)), 1, max_len) with u ~ U(0, ln max_len)."""
    u = torch.rand(batch, generator=gen, dtype=torch.float64) * math.log(max_len)
    return [int(min(max(round(math.exp(x)), 1), max_len)) for x in u.tolist()]


def quantize_e4m3_per_token(ckv_bf16: torch.Tensor):
    """bf16 [N, P, 512] -> (uint8 e4m3 codes [N, P, 512], fp32 scale [N, P])."""
    x = ckv_bf16.float()
    absmax = x.abs().amax(dim=-1)
    scale = absmax / E4M3_MAX
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    y = (x / safe.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX)
    y = torch.where((scale > 0).unsqueeze(-1), y, torch.zeros_like(y))
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def quantize_int8_per_token(ckv_bf16: torch.Tensor):
    """bf16 [N, P, 512] -> (int8 codes [N, P, 512], fp32 scale [N, P]): symmetric, one scale per
    token, scale = absmax / 127, code = round-half-even(x / scale) in fp32 (|code| <= 127)."""
    x = ckv_bf16.float()
    absmax = x.abs().amax(dim=-1)
    scale = absmax / 127.0
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    q = torch.round(x / safe.unsqueeze(-1)).clamp(-127, 127)
    q = torch.where((scale > 0).unsqueeze(-1), q, torch.zeros_like(q))
    return q.to(torch.int8), scale


def make_inputs(w: Workload, *, kv_lens=None, batch=None, h_q=None, page_size=None,
                pool_pages=None, seed=None, nan_fill=True, fp8=None, int8=False, f16=False) -> Inputs:
    """Draw one seeded batch.  Keyword overrides build smaller variants of a workload.  ``f16``
    rounds q_nope, q_pe, ckv and kpe to fp16 instead of bf16 (same draws, same order)."""
    B = batch if batch is not None else w.batch
    H = h_q if h_q is not None else w.h_q
    P = page_size if page_size is not None else w.page_size
    fp8 = w.fp8 if fp8 is None else fp8
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)

    if kv_lens is None:
        if w.kv_lens is not None and batch is None:
            kv_lens = list(w.kv_lens)
        elif w.ragged_max is not None:
            kv_lens = ragged_lengths(gen, B, w.ragged_max)
        else:
            kv_lens = [w.kv_len] * B
    kv_lens = [int(x) for x in kv_lens]
    assert len(kv_lens) == B
    n_pages = [(L + P - 1) // P for L in kv_lens]
    used = sum(n_pages)
    pool = pool_pages if pool_pages is not None else (w.pool_pages if (w.pool_pages and batch is None) else used)
    pool = max(pool, used, 1)

    perm = torch.randperm(pool, generator=gen).to(torch.int32)
    indptr = [0]
    for n in n_pages:
        indptr.append(indptr[-1] + n)
    kv_indptr = torch.tensor(indptr, dtype=torch.int32)
    kv_indices = perm[:used].clone()
    last = [(L - (n - 1) * P) if n > 0 else 0 for L, n in zip(kv_lens, n_pages)]
    kv_last_page_len = torch.tensor(last, dtype=torch.int32)

    dt = torch.float16 if f16 else torch.bfloat16
    q_nope = torch.randn(B, H, D_CKV, generator=gen).to(dt)
    q_pe = torch.randn(B, H, D_KPE, generator=gen).to(dt)
    ckv = torch.randn(pool, P, D_CKV, generator=gen).to(dt)
    kpe = torch.randn(pool, P, D_KPE, generator=gen).to(dt)

    if nan_fill:
        valid = torch.zeros(pool, P, dtype=torch.bool)
        for b in range(B):
            for j in range(n_pages[b]):
                pg = int(kv_indices[indptr[b] + j])
                valid[pg, : (P if j < n_pages[b] - 1 else last[b])] = True
        ckv[~valid] = float("nan")
        kpe[~valid] = float("nan")
    else:
        valid = None

    ckv_scale = None
    ckv_bf16 = None
    if int8:
        # INT8 cache: unused slots get the code -128 (never produced) and a NaN scale
        ckv_bf16 = ckv
        codes, ckv_scale = quantize_int8_per_token(torch.nan_to_num(ckv, nan=0.0))
        if valid is not None:
            codes[~valid] = -128
            ckv_scale[~valid] = float("nan")
        ckv = codes
    elif fp8:
        ckv_bf16 = ckv
        fin = torch.nan_to_num(ckv, nan=0.0)
        codes, ckv_scale = quantize_e4m3_per_token(fin)
        if valid is not None:
            codes[~valid] = 0x7F
            ckv_scale[~valid] = float("nan")
        ckv = codes

    return Inputs(w, q_nope, q_pe, ckv, kpe, kv_indptr, kv_indices, kv_last_page_len,
                  torch.tensor(kv_lens, dtype=torch.int64), ckv_scale, ckv_bf16)


def query_rows(inp: Inputs, qo_len: int, seed: int, f16: bool = False):
    """Queries for qo_len new tokens per request, from their own seeded generator:
    (q_nope [B * qo_len, H, 512], q_pe [B * qo_len, H, 64]) bf16 (fp16 with ``f16``), row
    b * qo_len + j being token j of request b."""
    gen = torch.Generator().manual_seed(seed)
    R = inp.batch * qo_len
    dt = torch.float16 if f16 else torch.bfloat16
    q_nope = torch.randn(R, inp.h_q, D_CKV, generator=gen).to(dt)
    q_pe = torch.randn(R, inp.h_q, D_KPE, generator=gen).to(dt)
    return q_nope, q_pe


def rope_table(max_pos: int, base: float = 10000.0) -> torch.Tensor:
    """fp32 [max_pos, 64]: cos(t * base^(-i / 32)) for pairs i = 0..31, then their sin (the
    usual rotary frequencies over the 64 rope dims)."""
    t = torch.arange(max_pos, dtype=torch.float64).unsqueeze(1)
    inv = base ** (-torch.arange(32, dtype=torch.float64) / 32.0)
    ang = t * inv
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(torch.float32)


def new_tokens(inp: Inputs, qo_len: int, seed: int, f16: bool = False):
    """The new tokens' inputs to the prologue, from their own seeded generator: pre-rotation
    q_pe [B * qo_len, H, 64], latent ckv [B * qo_len, 512] and pre-rotation kpe [B * qo_len, 64],
    all bf16 (fp16 with ``f16``)."""
    gen = torch.Generator().manual_seed(seed)
    R = inp.batch * qo_len
    dt = torch.float16 if f16 else torch.bfloat16
    q_pe = torch.randn(R, inp.h_q, D_KPE, generator=gen).to(dt)
    ckv = torch.randn(R, D_CKV, generator=gen).to(dt)
    kpe = torch.randn(R, D_KPE, generator=gen).to(dt)
    return q_pe, ckv, kpe


def algorithmic_bytes(inp: Inputs) -> int:
    """Bytes the method must move once: the KV tokens, q, out, lse and the page indices."""
    H = inp.h_q
    per_tok = (D_CKV + 4 + 2 * D_KPE) if inp.ckv_scale is not None else 2 * (D_CKV + D_KPE)
    L = int(inp.kv_lens.sum())
    n = int(inp.kv_indptr[-1])
    B = inp.batch
    return L * per_tok + B * (H * (D_CKV + D_KPE) * 2 + H * D_CKV * 4 + H * 4) + 4 * n + 8 * B


def algorithmic_flops(inp: Inputs) -> int:
    """2*H*L*(576 + 512): the QK^T and PV contractions; exp is not counted."""
    return 2 * inp.h_q * int(inp.kv_lens.sum()) * (D_CKV + D_KPE + D_CKV)


def layer_weights(seed: int, d_model: int = 2048, heads: int = 16, d_nope: int = 128, d_v: int = 128):
    """Synthetic weights of one MLA decode layer (DeepSeek-V2-Lite's sizes by default), bf16 on
    the CPU, from their own seeded generator: w_q [D, H, d_nope + 64], w_kv [D, 512],
    w_kpe [D, 64], w_uk [H, d_nope, 512], w_uv [H, 512, d_v], w_o [H * d_v, D]; each drawn
    gaussian and divided by the square root of its input width, so activations stay O(1)."""
    gen = torch.Generator().manual_seed(seed)

    def draw(*shape, fan_in):
        return (torch.randn(*shape, generator=gen) / fan_in ** 0.5).to(torch.bfloat16)

    import types
    return types.SimpleNamespace(
        w_q=draw(d_model, heads, d_nope + D_KPE, fan_in=d_model),
        w_kv=draw(d_model, D_CKV, fan_in=d_model),
        w_kpe=draw(d_model, D_KPE, fan_in=d_model),
        w_uk=draw(heads, d_nope, D_CKV, fan_in=d_nope),
        w_uv=draw(heads, D_CKV, d_v, fan_in=D_CKV),
        w_o=draw(heads * d_v, d_model, fan_in=heads * d_v),
    )


def layer_hidden(batch: int, seed: int, d_model: int = 2048) -> torch.Tensor:
    """The new tokens' hidden states x [B, D], bf16, from their own seeded generator."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(batch, d_model, generator=gen).to(torch.bfloat16)
