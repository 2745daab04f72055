"""The C-ABI library builds, loads without a GPU, and exports every function
declared in include/*.h; host-side argument checks return the documented codes."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
from mla_paged_kv_decode_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if lib_build.needs_build():
        lib_build.build()
    return mla.load()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    assert "mla_decode_plan" in names and "mla_decode_run" in names
    assert set(mla.EXPORTED) <= set(names)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    out = os.popen(f"nm -D --defined-only {mla.library_path()}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), f"{name} is not a defined dynamic symbol"


def test_status_strings(lib):
    for st in range(7):
        assert mla.mla_status_string(st)
    assert mla.mla_status_string(99) == "unknown status"


def _plan_rc(indptr, last, batch, h_q=16, page_size=16, sms=152, dtype=0):
    lib = mla.load()
    ip = np.ascontiguousarray(np.asarray(indptr, dtype=np.int32))
    lp = np.ascontiguousarray(np.asarray(last, dtype=np.int32))
    h = ctypes.c_void_p()
    rc = lib.mla_decode_plan(ip.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                             lp.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), batch, h_q, page_size, sms, dtype,
                             ctypes.byref(h))
    if rc == 0:
        lib.mla_plan_destroy(h)
    return rc


def test_plan_argument_checks(lib):
    assert _plan_rc([0, 1, 3], [5, 16], 2) == mla.MLA_OK
    assert _plan_rc([0, 1, 3], [0, 16], 2) == mla.MLA_ERR_INVALID_ARG      # last_page_len 0 on a non-empty request
    assert _plan_rc([0, 1, 3], [5, 17], 2) == mla.MLA_ERR_INVALID_ARG      # last_page_len > page_size
    assert _plan_rc([0, 3, 1], [5, 5], 2) == mla.MLA_ERR_INVALID_ARG       # indptr decreasing
    assert _plan_rc([1, 3], [5], 1) == mla.MLA_ERR_INVALID_ARG             # indptr[0] != 0
    assert _plan_rc([0, 1], [5], 0) == mla.MLA_ERR_INVALID_ARG             # batch 0
    assert _plan_rc([0, 1], [5], 1, sms=0) == mla.MLA_ERR_INVALID_ARG
    assert _plan_rc([0, 1], [5], 1, h_q=8) == mla.MLA_ERR_UNSUPPORTED
    assert _plan_rc([0, 1], [5], 1, page_size=8) == mla.MLA_ERR_UNSUPPORTED
    assert _plan_rc([0, 0, 1], [0, 5], 2) == mla.MLA_OK                    # an empty request is allowed
    assert _plan_rc([0, 1], [5], 1, dtype=7) == mla.MLA_ERR_INVALID_ARG


def test_run_and_commit_reject_bad_arguments_without_touching_a_gpu(lib):
    plan = mla.mla_decode_plan(torch.tensor([0, 2]), torch.tensor([7]), 1, 16, 16, 152)
    assert plan.workspace_bytes % 256 == 0 and plan.workspace_bytes > 0
    vp = ctypes.c_void_p
    # NULL workspace / unaligned workspace / too small: rejected on the host
    assert lib.mla_decode_plan_commit(plan.handle, None, 1 << 20, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_plan_commit(plan.handle, vp(4096 + 16), 1 << 20, None) == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_plan_commit(plan.handle, vp(4096), 16, None) == mla.MLA_ERR_WORKSPACE_TOO_SMALL
    # run before commit
    fake = vp(1 << 20)
    rc = lib.mla_decode_run(plan.handle, fake, fake, fake, None, fake, 4, fake, fake, fake, ctypes.c_float(0.1),
                            fake, fake, vp(1 << 21), None)
    assert rc == mla.MLA_ERR_NOT_COMMITTED
    rc = lib.mla_decode_run(plan.handle, None, fake, fake, None, fake, 4, fake, fake, fake, ctypes.c_float(0.1),
                            fake, fake, vp(1 << 21), None)
    assert rc == mla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_plan_workspace_bytes(None) == 0
    assert lib.mla_plan_num_ctas(None) == 0


def test_fp8_plan_and_run_checks(lib):
    # the e4m3 cache is served for every supported head count; others are refused at plan time
    for h_q in (16, 32, 64, 128):
        assert _plan_rc([0, 1], [5], 1, h_q=h_q, dtype=mla.MLA_KV_FP8_E4M3) == mla.MLA_OK
    for h_q in (8, 48, 256):
        assert _plan_rc([0, 1], [5], 1, h_q=h_q, dtype=mla.MLA_KV_FP8_E4M3) == mla.MLA_ERR_UNSUPPORTED
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    plan = mla.mla_decode_plan(torch.tensor([0, 2]), torch.tensor([7]), 1, 16, 16, 152, mla.MLA_KV_FP8_E4M3)
    # an 8-bit plan needs the scales, 16-byte aligned; a bf16 plan must not get any
    for scale in (None, vp((1 << 20) + 4)):
        rc = lib.mla_decode_run(plan.handle, fake, fake, fake, scale, fake, 4, fake, fake, fake, ctypes.c_float(0.1),
                                fake, fake, vp(1 << 21), None)
        assert rc == mla.MLA_ERR_INVALID_ARG
    plan16 = mla.mla_decode_plan(torch.tensor([0, 2]), torch.tensor([7]), 1, 16, 16, 152)
    rc = lib.mla_decode_run(plan16.handle, fake, fake, fake, fake, fake, 4, fake, fake, fake, ctypes.c_float(0.1),
                            fake, fake, vp(1 << 21), None)
    assert rc == mla.MLA_ERR_INVALID_ARG


def test_prologue_rejects_bad_arguments_without_touching_a_gpu(lib):
    """Every case fails a host check before any CUDA call (the pointers are never dereferenced)."""
    vp = ctypes.c_void_p
    f = vp(1 << 20)

    def rc(batch=1, qo_len=1, h_q=16, P=16, dtype=mla.MLA_KV_BF16, scale=None, max_pos=8, num_pages=4, ckv_new=f,
           q_in=f):
        return lib.mla_decode_prologue(batch, qo_len, h_q, P, dtype, 1, q_in, f, ckv_new, f, f, max_pos, f, f, f, f,
                                       scale, f, num_pages, None)

    assert rc(batch=0) == mla.MLA_ERR_INVALID_ARG
    assert rc(qo_len=0) == mla.MLA_ERR_INVALID_ARG
    assert rc(qo_len=65) == mla.MLA_ERR_INVALID_ARG
    assert rc(h_q=0) == mla.MLA_ERR_INVALID_ARG
    assert rc(max_pos=0) == mla.MLA_ERR_INVALID_ARG
    assert rc(num_pages=0) == mla.MLA_ERR_INVALID_ARG
    assert rc(P=24) == mla.MLA_ERR_UNSUPPORTED
    assert rc(dtype=7) == mla.MLA_ERR_INVALID_ARG
    assert rc(dtype=mla.MLA_KV_FP8_E4M3) == mla.MLA_ERR_INVALID_ARG              # 8-bit cache without scales
    assert rc(dtype=mla.MLA_KV_BF16, scale=f) == mla.MLA_ERR_INVALID_ARG         # bf16 cache with scales
    assert rc(ckv_new=vp((1 << 20) + 4)) == mla.MLA_ERR_INVALID_ARG               # latent rows need 8-byte alignment
    assert rc(q_in=None) == mla.MLA_ERR_INVALID_ARG


def test_header_is_plain_c(tmp_path):
    """include/mla_decode.h compiles as C99 (no C++ in the ABI) and as C++."""
    src = tmp_path / "use.c"
    src.write_text('#include "mla_decode.h"\nint main(void) { mla_plan_t p = 0; (void)p; return (int)MLA_OK; }\n')
    inc = os.path.join(ROOT, "include")
    for lang, std in (("c", "-std=c99"), ("c++", "-std=c++17")):
        r = os.system(f"gcc -x {lang} {std} -Wall -Werror -pedantic -fsyntax-only -I{inc} {src} 2>/dev/null")
        assert r == 0, f"the header does not compile as {lang}"
