"""TEST INFRASTRUCTURE: the fp64 CPU oracle for MLA paged-KV decode.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its cpu
baseline and ``--impl reference`` arm) may import this package.  The product
path (``mla_paged_kv_decode_gb300``) never does, and shares no code with it.

Two independent implementations live here:
  * ``mla_decode`` / ``mla_decode_range`` / ``merge`` / ``e4m3_*``: plain C in
    fp64 (``mla_oracle.c``), the definition written out loop by loop;
  * ``brute.brute_force``: torch fp64, materialising K and V by Python
    indexing and calling ``torch.softmax`` / ``torch.logsumexp``, used to pin
    the C oracle on small shapes.
See ``mla_oracle.c`` for the definition and the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(out_path: str = _LIB_PATH, plant: int = 0) -> str:
    """Compile the oracle (gcc, -O2, OpenMP).  ``plant`` != 0 builds a copy with a
    deliberate mistake, used only by the test that proves the pins catch it."""
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", f"-DORACLE_PLANT={int(plant)}",
           _SRC, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


def _bind(lib):
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.oracle_mla_decode.restype = ctypes.c_int
    lib.oracle_mla_decode.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_void_p, i32p, i32p, i32p,
                                      ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_mla_decode_range.restype = ctypes.c_int
    lib.oracle_mla_decode_range.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_void_p, i32p, i32p,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                            ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_merge.restype = None
    lib.oracle_merge.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_f16_decode.restype = ctypes.c_double
    lib.oracle_f16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
    return lib


def load(path: Optional[str] = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _u16(t: torch.Tensor) -> np.ndarray:
    assert t.dtype in (torch.bfloat16, torch.float16)
    return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(t) -> np.ndarray:
    return np.ascontiguousarray(torch.as_tensor(t).to(torch.int32).numpy())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _ip(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _cache_arrays(ckv, ckv_scale):
    """(codes or 16-bit bits, cache kind: 0 bf16, 1 e4m3 codes (uint8), 2 int8 codes, 3 fp16, scales)."""
    if ckv.dtype in (torch.uint8, torch.int8):
        assert ckv_scale is not None, "8-bit cache needs its per-token scales"
        return np.ascontiguousarray(ckv.contiguous().view(torch.uint8).numpy()), \
            (1 if ckv.dtype == torch.uint8 else 2), np.ascontiguousarray(ckv_scale.contiguous().to(torch.float32).numpy())
    return _u16(ckv), (3 if ckv.dtype == torch.float16 else 0), None


def _check_16bit(q_nope, q_pe, ckv, kpe):
    """fp16 inputs are all fp16 (the cache kind decides how q and kpe are read)."""
    f16 = ckv.dtype == torch.float16
    for t in (q_nope, q_pe, kpe):
        assert (t.dtype == torch.float16) == f16, "q, ckv and kpe must all be fp16, or none of them"


def mla_decode(q_nope, q_pe, ckv, kpe, kv_indices, kv_indptr, kv_last_page_len, sm_scale,
               ckv_scale=None, threads: int = 0, lib=None):
    """fp64 oracle.  CPU tensors in the library's layout; returns (out [B,H,512], lse [B,H])
    as float64 torch tensors."""
    lib = lib or load()
    B, H, _ = q_nope.shape
    P = ckv.shape[1]
    _check_16bit(q_nope, q_pe, ckv, kpe)
    qn, qp, kp = _u16(q_nope), _u16(q_pe), _u16(kpe)
    ck, is8, sc = _cache_arrays(ckv, ckv_scale)
    ind, iptr, last = _i32(kv_indices), _i32(kv_indptr), _i32(kv_last_page_len)
    out = np.zeros((B, H, 512), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    rc = lib.oracle_mla_decode(B, H, P, _ptr(qn), _ptr(qp), _ptr(ck), is8,
                               _ptr(sc) if sc is not None else None, _ptr(kp),
                               _ip(ind), _ip(iptr), _ip(last), float(sm_scale),
                               _ptr(out), _ptr(lse), int(threads))
    if rc != 0:
        raise MemoryError("oracle_mla_decode failed")
    return torch.from_numpy(out), torch.from_numpy(lse)


def mla_decode_range(b, t_begin, t_end, q_nope, q_pe, ckv, kpe, kv_indices, kv_indptr, sm_scale,
                     ckv_scale=None, lib=None):
    """Partial (out [H,512], lse [H]) of request b over its tokens [t_begin, t_end)."""
    lib = lib or load()
    B, H, _ = q_nope.shape
    P = ckv.shape[1]
    _check_16bit(q_nope, q_pe, ckv, kpe)
    qn, qp, kp = _u16(q_nope), _u16(q_pe), _u16(kpe)
    ck, is8, sc = _cache_arrays(ckv, ckv_scale)
    ind, iptr = _i32(kv_indices), _i32(kv_indptr)
    out = np.zeros((H, 512), dtype=np.float64)
    lse = np.zeros((H,), dtype=np.float64)
    rc = lib.oracle_mla_decode_range(H, P, int(b), _ptr(qn), _ptr(qp), _ptr(ck), is8,
                                     _ptr(sc) if sc is not None else None, _ptr(kp), _ip(ind), _ip(iptr),
                                     int(t_begin), int(t_end), float(sm_scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise MemoryError("oracle_mla_decode_range failed")
    return torch.from_numpy(out), torch.from_numpy(lse)


def mla_decode_rows(q_nope, q_pe, ckv, kpe, kv_indices, kv_indptr, kv_last_page_len, sm_scale, qo_len: int,
                    causal: bool, ckv_scale=None, lib=None):
    """Several query tokens per request.  q_nope [B * qo_len, H, 512], q_pe [B * qo_len, H, 64];
    row r = b * qo_len + j is query token j of request b, the new tokens being the last qo_len
    of its L_b cached tokens.  The row attends to the first L_b tokens, or, causal, to the first
    max(0, L_b - (qo_len - 1 - j)): each new token sees the cache up to itself.  Returns
    (out [B * qo_len, H, 512], lse [B * qo_len, H]) in fp64; a row with no tokens gets 0, -inf.
    Each row is the definition over its token prefix (``mla_decode_range`` of request b's pages)."""
    lib = lib or load()
    R, H, _ = q_nope.shape
    P = ckv.shape[1]
    B = R // qo_len
    assert B * qo_len == R
    indptr = [int(x) for x in kv_indptr]
    out = torch.zeros(R, H, 512, dtype=torch.float64)
    lse = torch.full((R, H), float("-inf"), dtype=torch.float64)
    for b in range(B):
        n = indptr[b + 1] - indptr[b]
        L = (n - 1) * P + int(kv_last_page_len[b]) if n > 0 else 0
        pages = kv_indices[indptr[b]:indptr[b + 1]]
        one = torch.tensor([0, n], dtype=torch.int32)
        for j in range(qo_len):
            r = b * qo_len + j
            Lr = max(0, L - (qo_len - 1 - j)) if causal else L
            if Lr == 0:
                continue
            o, l = mla_decode_range(0, 0, Lr, q_nope[r:r + 1], q_pe[r:r + 1], ckv, kpe, pages, one, sm_scale,
                                    ckv_scale=ckv_scale, lib=lib)
            out[r], lse[r] = o, l
    return out, lse


def rope_f64(x, cos, sin, interleaved: bool):
    """Rotate the 32 pairs of the last (64) dim of x in fp64: pair i is dims (2i, 2i + 1)
    when interleaved, else (i, i + 32); (a, b) -> (a cos_i - b sin_i, a sin_i + b cos_i)."""
    x = torch.as_tensor(x).to(torch.float64)
    c = torch.as_tensor(cos).to(torch.float64)
    s = torch.as_tensor(sin).to(torch.float64)
    ia = torch.arange(32) * 2 if interleaved else torch.arange(32)
    ib = ia + 1 if interleaved else ia + 32
    a, b = x[..., ia], x[..., ib]
    out = x.clone()
    out[..., ia] = a * c - b * s
    out[..., ib] = a * s + b * c
    return out


def decode_prologue(q_pe, ckv_new, kpe_new, rope_cos_sin, kv_indices, kv_indptr, kv_last_page_len, qo_len: int,
                    interleaved: bool, ckv_cache, kpe_cache, ckv_scale=None, lib=None):
    """The decode prologue on CPU tensors; returns new (q_pe_out, ckv_cache, kpe_cache, ckv_scale)
    and leaves the inputs untouched.  Row r = b * qo_len + j is new token j of request b, at
    position t = L_b - qo_len + j (the new tokens are the last qo_len of the cache), page
    kv_indices[kv_indptr[b] + t // P], slot t % P; a row with t < 0 or t >= max_pos is skipped.
    q_pe and kpe are rotated (``rope_f64``, then rounded to their own 16-bit type); ckv is copied,
    or for the e4m3 cache quantised with s = absmax / 448 and codes e4m3(x / s), both in fp32 (the
    precision the quantised code is decided in), ``e4m3_encode`` rounding to nearest even, or for
    the INT8 cache with s = absmax / 127 and codes x / s rounded half to even within +-127."""
    lib = lib or load()
    P = ckv_cache.shape[1]
    num_pages = ckv_cache.shape[0]
    max_pos = rope_cos_sin.shape[0]
    q_out, ckv, kpe = q_pe.clone(), ckv_cache.clone(), kpe_cache.clone()
    sc = ckv_scale.clone() if ckv_scale is not None else None
    indptr = [int(x) for x in kv_indptr]
    for r in range(q_pe.shape[0]):
        b, j = divmod(r, qo_len)
        n = indptr[b + 1] - indptr[b]
        L = (n - 1) * P + int(kv_last_page_len[b]) if n > 0 else 0
        t = L - qo_len + j
        if t < 0 or t >= max_pos:
            continue
        c, s = rope_cos_sin[t, :32], rope_cos_sin[t, 32:]
        q_out[r] = rope_f64(q_pe[r], c, s, interleaved).to(q_pe.dtype)
        page = int(kv_indices[indptr[b] + t // P])
        if not 0 <= page < num_pages:
            continue
        slot = t % P
        kpe[page, slot] = rope_f64(kpe_new[r], c, s, interleaved).to(kpe.dtype)
        if ckv.dtype == torch.int8:
            # INT8: s = absmax / 127 and codes x / s rounded half to even, in fp32
            x = ckv_new[r].to(torch.float32).numpy()
            scale = np.float32(np.abs(x).max()) / np.float32(127.0)
            if scale > 0:
                y = np.rint((x / scale).astype(np.float32))
                ckv[page, slot] = torch.from_numpy(np.clip(y, -127, 127).astype(np.int8))
            else:
                ckv[page, slot] = 0
            sc[page, slot] = float(scale)
        elif ckv.dtype == torch.uint8:
            x = ckv_new[r].to(torch.float32).numpy()
            scale = np.float32(np.abs(x).max()) / np.float32(448.0)
            if scale > 0:
                y = np.clip(x / scale, np.float32(-448.0), np.float32(448.0)).astype(np.float32)
                ckv[page, slot] = torch.from_numpy(e4m3_encode(y, lib=lib))
            else:
                ckv[page, slot] = 0
            sc[page, slot] = float(scale)
        else:
            ckv[page, slot] = ckv_new[r]
    return q_out, ckv, kpe, sc


def merge(o_parts, lse_parts, lib=None):
    """Merge k partials [k,H,D] / [k,H] (fixed order) -> (out [H,D], lse [H])."""
    lib = lib or load()
    o = np.ascontiguousarray(torch.as_tensor(o_parts, dtype=torch.float64).numpy())
    s = np.ascontiguousarray(torch.as_tensor(lse_parts, dtype=torch.float64).numpy())
    k, H, D = o.shape
    out = np.zeros((H, D), dtype=np.float64)
    lse = np.zeros((H,), dtype=np.float64)
    lib.oracle_merge(k, H, D, _ptr(o), _ptr(s), _ptr(out), _ptr(lse))
    return torch.from_numpy(out), torch.from_numpy(lse)


def f16_decode(bits, lib=None) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64 (the oracle's own decoder)."""
    lib = lib or load()
    return np.array([lib.oracle_f16_decode(int(b)) for b in np.asarray(bits).ravel()], dtype=np.float64)


def e4m3_decode(codes, lib=None) -> np.ndarray:
    lib = lib or load()
    return np.array([lib.oracle_e4m3_decode(int(c)) for c in np.asarray(codes).ravel()], dtype=np.float64)


def e4m3_encode(values, lib=None) -> np.ndarray:
    lib = lib or load()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in np.asarray(values, dtype=np.float64).ravel()],
                    dtype=np.uint8)


def decode_inputs(inp, threads: int = 0, use_bf16_cache: bool = False):
    """Run the oracle on a ``workloads.Inputs``.  ``use_bf16_cache`` runs an 8-bit
    workload on the bf16 cache it was quantised from."""
    if inp.ckv_scale is not None and not use_bf16_cache:
        return mla_decode(inp.q_nope, inp.q_pe, inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr,
                          inp.kv_last_page_len, inp.sm_scale, ckv_scale=inp.ckv_scale, threads=threads)
    ckv = inp.ckv_bf16 if inp.ckv_scale is not None else inp.ckv
    return mla_decode(inp.q_nope, inp.q_pe, ckv, inp.kpe, inp.kv_indices, inp.kv_indptr,
                      inp.kv_last_page_len, inp.sm_scale, threads=threads)


def decode_subset(inp, requests, threads: int = 0, use_bf16_cache: bool = False):
    """Oracle on a subset of a ``workloads.Inputs`` batch: the same cache, with q and
    the page table sliced to ``requests``."""
    idx = torch.as_tensor(list(requests), dtype=torch.long)
    indptr = inp.kv_indptr.long()
    pieces = [inp.kv_indices[indptr[b]:indptr[b + 1]] for b in requests]
    sub_ind = torch.cat(pieces) if pieces else inp.kv_indices[:0]
    sub_ptr = torch.zeros(len(pieces) + 1, dtype=torch.int32)
    if pieces:
        sub_ptr[1:] = torch.cumsum(torch.tensor([len(p) for p in pieces]), 0).to(torch.int32)
    ckv, scale = inp.ckv, inp.ckv_scale
    if use_bf16_cache and inp.ckv_bf16 is not None:
        ckv, scale = inp.ckv_bf16, None
    return mla_decode(inp.q_nope[idx], inp.q_pe[idx], ckv, inp.kpe, sub_ind, sub_ptr, inp.kv_last_page_len[idx],
                      inp.sm_scale, ckv_scale=scale, threads=threads)
