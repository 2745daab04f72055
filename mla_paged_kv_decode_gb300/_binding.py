"""ctypes binding of include/mla_decode.h.  Argument marshalling only: every
step of the decode runs in the CUDA library.  Functions keep the C names.

Tensors are torch tensors on the device the library runs on (host int32
tensors for the plan's index arrays).  Streams default to torch's current
stream.  A status other than MLA_OK raises ``MLAError``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

from . import build as _build

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE_TOO_SMALL = 3
MLA_ERR_CUDA = 4
MLA_ERR_DEVICE_TIMEOUT = 5
MLA_ERR_NOT_COMMITTED = 6

MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3 = 1
MLA_KV_INT8 = 2
MLA_KV_F16 = 3

MLA_OUT_F32 = 0
MLA_OUT_BF16 = 1

EXPORTED = (
    "mla_decode_plan", "mla_decode_plan_workspace_bytes", "mla_decode_plan_commit", "mla_decode_run",
    "mla_decode_device_status", "mla_plan_num_ctas", "mla_plan_num_segments", "mla_plan_num_partials",
    "mla_plan_heads_per_cta", "mla_plan_get_segments", "mla_plan_destroy", "mla_status_string",
    "mla_plan_num_launches", "mla_decode_run_noalloc", "mla_decode_noalloc_max_workspace_bytes",
    "mla_plan_segment_cost_tiles", "mla_plan_num_units", "mla_decode_plan_ex", "mla_plan_num_rows",
    "mla_decode_prologue",
)

_lib = None


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {mla_status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None):
    """Load the compiled library.  Raises ImportError if it has not been built:
    there is no fallback implementation."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it with `python -m mla_paged_kv_decode_gb300.build` "
                          "(or __graft_entry__.build()); there is no CPU or PyTorch fallback")
    lib = ctypes.CDLL(p)
    vp, i32p, sz = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_size_t
    lib.mla_decode_plan.restype = ctypes.c_int
    lib.mla_decode_plan.argtypes = [i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.POINTER(vp)]
    lib.mla_decode_plan_ex.restype = ctypes.c_int
    lib.mla_decode_plan_ex.argtypes = [i32p, i32p] + [ctypes.c_int] * 8 + [ctypes.POINTER(vp)]
    lib.mla_decode_prologue.restype = ctypes.c_int
    lib.mla_decode_prologue.argtypes = [ctypes.c_int] * 6 + [vp] * 5 + [ctypes.c_int] + [vp] * 6 + [ctypes.c_int, vp]
    lib.mla_decode_plan_workspace_bytes.restype = sz
    lib.mla_decode_plan_workspace_bytes.argtypes = [vp]
    lib.mla_decode_plan_commit.restype = ctypes.c_int
    lib.mla_decode_plan_commit.argtypes = [vp, vp, sz, vp]
    lib.mla_decode_run.restype = ctypes.c_int
    lib.mla_decode_run.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp]
    lib.mla_decode_run_noalloc.restype = ctypes.c_int
    lib.mla_decode_run_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp, ctypes.c_float, vp, vp,
                                           vp]
    lib.mla_decode_noalloc_max_workspace_bytes.restype = sz
    lib.mla_decode_noalloc_max_workspace_bytes.argtypes = []
    lib.mla_plan_num_launches.restype = ctypes.c_int
    lib.mla_plan_num_launches.argtypes = [vp]
    lib.mla_decode_device_status.restype = ctypes.c_int
    lib.mla_decode_device_status.argtypes = [vp, vp, vp]
    for name in ("mla_plan_num_ctas", "mla_plan_num_segments", "mla_plan_num_partials", "mla_plan_heads_per_cta",
                 "mla_plan_segment_cost_tiles", "mla_plan_num_units", "mla_plan_num_rows"):
        getattr(lib, name).restype = ctypes.c_int
        getattr(lib, name).argtypes = [vp]
    lib.mla_plan_get_segments.restype = ctypes.c_int
    lib.mla_plan_get_segments.argtypes = [vp, i32p, i32p]
    lib.mla_plan_destroy.restype = None
    lib.mla_plan_destroy.argtypes = [vp]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [ctypes.c_int]
    if path is None:
        _lib = lib
    return lib


def mla_status_string(status: int) -> str:
    return load().mla_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MLA_OK:
        raise MLAError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.is_contiguous(), "tensors must be contiguous"
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Plan:
    """Owns an mla_plan_t handle (destroyed with the object)."""

    def __init__(self, handle, batch, h_q, page_size, kv_dtype, qo_len=1, causal=False, out_dtype=MLA_OUT_F32):
        self.handle = handle
        self.batch, self.h_q, self.page_size, self.kv_dtype = batch, h_q, page_size, kv_dtype
        self.qo_len, self.causal, self.out_dtype = qo_len, causal, out_dtype

    @property
    def workspace_bytes(self) -> int:
        return mla_decode_plan_workspace_bytes(self)

    def __del__(self):
        if getattr(self, "handle", None) is not None and _lib is not None:
            _lib.mla_plan_destroy(self.handle)
            self.handle = None


def mla_decode_plan(kv_indptr, kv_last_page_len, batch: int, h_q: int, page_size: int, num_sms: int,
                    kv_dtype: int = MLA_KV_BF16) -> Plan:
    lib = load()
    ip = np.ascontiguousarray(torch.as_tensor(kv_indptr).cpu().to(torch.int32).numpy())
    lp = np.ascontiguousarray(torch.as_tensor(kv_last_page_len).cpu().to(torch.int32).numpy())
    h = ctypes.c_void_p()
    st = lib.mla_decode_plan(ip.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                             lp.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(batch), int(h_q),
                             int(page_size), int(num_sms), int(kv_dtype), ctypes.byref(h))
    _check(st, "mla_decode_plan")
    return Plan(h, batch, h_q, page_size, kv_dtype)


def mla_decode_plan_ex(kv_indptr, kv_last_page_len, batch: int, qo_len: int, causal: bool, h_q: int,
                       page_size: int, num_sms: int, kv_dtype: int = MLA_KV_BF16,
                       out_dtype: int = MLA_OUT_F32) -> Plan:
    lib = load()
    ip = np.ascontiguousarray(torch.as_tensor(kv_indptr).cpu().to(torch.int32).numpy())
    lp = np.ascontiguousarray(torch.as_tensor(kv_last_page_len).cpu().to(torch.int32).numpy())
    h = ctypes.c_void_p()
    st = lib.mla_decode_plan_ex(ip.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                lp.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(batch), int(qo_len),
                                int(bool(causal)), int(h_q), int(page_size), int(num_sms), int(kv_dtype),
                                int(out_dtype), ctypes.byref(h))
    _check(st, "mla_decode_plan_ex")
    return Plan(h, batch, h_q, page_size, kv_dtype, qo_len, bool(causal), out_dtype)


def mla_decode_prologue(batch: int, qo_len: int, h_q: int, page_size: int, kv_dtype: int, rope_interleaved: bool,
                        q_pe_in, q_pe_out, ckv_new, kpe_new, rope_cos_sin, kv_indices, kv_indptr, kv_last_page_len,
                        ckv_cache, ckv_scale, kpe_cache, stream=None):
    _check(load().mla_decode_prologue(int(batch), int(qo_len), int(h_q), int(page_size), int(kv_dtype),
                                      int(bool(rope_interleaved)), _ptr(q_pe_in), _ptr(q_pe_out), _ptr(ckv_new),
                                      _ptr(kpe_new), _ptr(rope_cos_sin), int(rope_cos_sin.shape[0]), _ptr(kv_indices),
                                      _ptr(kv_indptr), _ptr(kv_last_page_len), _ptr(ckv_cache), _ptr(ckv_scale),
                                      _ptr(kpe_cache), int(ckv_cache.shape[0]), _stream(stream)),
           "mla_decode_prologue")


def mla_plan_num_rows(plan: Plan) -> int:
    return int(load().mla_plan_num_rows(plan.handle))


def mla_decode_plan_workspace_bytes(plan: Plan) -> int:
    return int(load().mla_decode_plan_workspace_bytes(plan.handle))


def mla_decode_plan_commit(plan: Plan, workspace: torch.Tensor, stream=None):
    _check(load().mla_decode_plan_commit(plan.handle, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream)), "mla_decode_plan_commit")


def mla_decode_run(plan: Plan, q_nope, q_pe, ckv_cache, ckv_scale, kpe_cache, kv_indices, kv_indptr,
                   kv_last_page_len, sm_scale: float, out, lse, workspace, stream=None, num_pages=None):
    npages = int(ckv_cache.shape[0]) if num_pages is None else int(num_pages)
    _check(load().mla_decode_run(plan.handle, _ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(ckv_scale),
                                 _ptr(kpe_cache), npages, _ptr(kv_indices), _ptr(kv_indptr), _ptr(kv_last_page_len),
                                 float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), _stream(stream)),
           "mla_decode_run")


def mla_decode_run_noalloc(plan: Plan, q_nope, q_pe, ckv_cache, ckv_scale, kpe_cache, kv_indices, kv_indptr,
                           kv_last_page_len, sm_scale: float, out, lse, stream=None, num_pages=None):
    """mla_decode_run without a workspace: the library's fixed device array is used instead
    (for callers that cannot allocate device memory; calls that overlap on the GPU race)."""
    npages = int(ckv_cache.shape[0]) if num_pages is None else int(num_pages)
    _check(load().mla_decode_run_noalloc(plan.handle, _ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(ckv_scale),
                                         _ptr(kpe_cache), npages, _ptr(kv_indices), _ptr(kv_indptr),
                                         _ptr(kv_last_page_len), float(sm_scale), _ptr(out), _ptr(lse), _stream(stream)),
           "mla_decode_run_noalloc")


def mla_decode_noalloc_max_workspace_bytes() -> int:
    return int(load().mla_decode_noalloc_max_workspace_bytes())


def mla_plan_num_launches(plan: Plan) -> int:
    return int(load().mla_plan_num_launches(plan.handle))


def mla_decode_device_status(plan: Plan, workspace, stream=None) -> int:
    return int(load().mla_decode_device_status(plan.handle, _ptr(workspace), _stream(stream)))


def mla_plan_num_ctas(plan: Plan) -> int:
    return int(load().mla_plan_num_ctas(plan.handle))


def mla_plan_num_segments(plan: Plan) -> int:
    return int(load().mla_plan_num_segments(plan.handle))


def mla_plan_num_partials(plan: Plan) -> int:
    return int(load().mla_plan_num_partials(plan.handle))


def mla_plan_heads_per_cta(plan: Plan) -> int:
    return int(load().mla_plan_heads_per_cta(plan.handle))


def mla_plan_num_units(plan: Plan) -> int:
    return int(load().mla_plan_num_units(plan.handle))


def mla_plan_segment_cost_tiles(plan: Plan) -> int:
    return int(load().mla_plan_segment_cost_tiles(plan.handle))


def mla_plan_get_segments(plan: Plan):
    """-> (segments int32 [n, 4] = (request, token_begin, token_end, slot), unit_ptr int32 [units + 1])"""
    lib = load()
    n = lib.mla_plan_num_segments(plan.handle)
    units = lib.mla_plan_num_units(plan.handle)
    seg = np.zeros((max(n, 1), 4), dtype=np.int32)
    uptr = np.zeros(units + 1, dtype=np.int32)
    lib.mla_plan_get_segments(plan.handle, seg.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                              uptr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    return seg[:n], uptr
