"""A bounded device wait that runs out, made without any fault.

Every mbarrier wait in the kernels gives up after a time limit: the waiter raises the CTA's abort
flag, records 0x100 | its wait site in the status word, the producers wait (bounded) for their
copies in flight, and the kernel returns.  mla_decode_device_status then reports
MLA_ERR_DEVICE_TIMEOUT.  This test builds a test copy of the library with a 2 ms limit and a
hook that makes the narrow-head kernel's CTA 0 withhold the copy of its first ring stage -- a
barrier nothing completes -- and checks:

* the run returns, the status word names the site of a wait that ran out because of the
  withheld stage (whichever reached the limit first), and mla_decode_device_status reports
  MLA_ERR_DEVICE_TIMEOUT (and clears the word);
* after a re-commit (which resets the workspace's counters) a run without the hook gives the
  same bits as a clean run, and the status is MLA_OK;
* the same for mla_decode_run_noalloc, whose status word is read with a NULL workspace.
"""
import ctypes

import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
from mla_paged_kv_decode_gb300 import build as lib_build
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

# the waits the withheld stage can make run out; the first to reach the limit records its site
SITES = (21,   # the producer waiting for the withheld stage's release before refilling it
         22,   # a compute group waiting for the stage to land
         23,   # the other token group waiting for the stage's release before its own tile
         24)   # a last-arriving piece (in any CTA) waiting for the other pieces' partials


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    path = str(tmp_path_factory.mktemp("mla_test_build") / "libmla_decode_waitlimit.so")
    lib_build.build(out=path, extra=("-DMLA_TEST_HOOKS", "-DMLA_WAIT_LIMIT_NS=2000000ull"))
    lib = mla.load(path)   # a separate handle: the product library stays loaded as it is
    lib.mla_debug_set_withhold.restype = None
    lib.mla_debug_set_withhold.argtypes = [ctypes.c_void_p, ctypes.c_int]
    return lib


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_withheld_stage_times_out_and_the_next_run_is_clean(lib):
    inp = make_inputs(WORKLOADS["tiny"], kv_lens=[3000, 5, 700, 4096, 129], batch=5, h_q=16, page_size=64, seed=111)
    d = inp.to("cuda")
    i32p = ctypes.POINTER(ctypes.c_int32)
    ip = inp.kv_indptr.to(torch.int32).contiguous()
    lp = inp.kv_last_page_len.to(torch.int32).contiguous()
    handle = ctypes.c_void_p()
    rc = lib.mla_decode_plan(ctypes.cast(ip.data_ptr(), i32p), ctypes.cast(lp.data_ptr(), i32p), inp.batch, inp.h_q,
                             inp.page_size, mla.num_sms(), mla.MLA_KV_BF16, ctypes.byref(handle))
    assert rc == mla.MLA_OK
    assert lib.mla_plan_num_partials(handle) > 0   # split pieces: merges wait across CTAs too
    nbytes = lib.mla_decode_plan_workspace_bytes(handle)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.empty(inp.batch, inp.h_q, 512, device="cuda")
    lse = torch.empty(inp.batch, inp.h_q, device="cuda")

    def run(noalloc=False):
        args = [handle, _vp(d.q_nope), _vp(d.q_pe), _vp(d.ckv), None, _vp(d.kpe), inp.num_pages, _vp(d.kv_indices),
                _vp(d.kv_indptr), _vp(d.kv_last_page_len), ctypes.c_float(inp.sm_scale), _vp(out), _vp(lse)]
        rc = lib.mla_decode_run_noalloc(*args, stream) if noalloc else lib.mla_decode_run(*args, _vp(ws), stream)
        assert rc == mla.MLA_OK
        torch.cuda.synchronize()

    try:
        assert lib.mla_decode_plan_commit(handle, _vp(ws), nbytes, stream) == mla.MLA_OK
        run()
        assert lib.mla_decode_device_status(handle, _vp(ws), stream) == mla.MLA_OK
        clean_out, clean_lse = out.clone(), lse.clone()

        # CTA 0 withholds its first stage: the wait on it runs out after 2 ms
        lib.mla_debug_set_withhold(handle, 1)
        run()
        word = int(ws[:4].view(torch.int32).item())
        assert word in tuple(0x100 | site for site in SITES), hex(word)
        assert lib.mla_decode_device_status(handle, _vp(ws), stream) == mla.MLA_ERR_DEVICE_TIMEOUT
        assert int(ws[:4].view(torch.int32).item()) == 0   # read once, then cleared

        # re-commit (the counters the aborted run left), then a normal run: the clean bits
        lib.mla_debug_set_withhold(handle, 0)
        assert lib.mla_decode_plan_commit(handle, _vp(ws), nbytes, stream) == mla.MLA_OK
        out.fill_(float("nan"))
        run()
        assert lib.mla_decode_device_status(handle, _vp(ws), stream) == mla.MLA_OK
        assert torch.equal(out, clean_out) and torch.equal(lse, clean_lse)

        # the no-allocation entry point: the status word of its fixed array (NULL workspace)
        lib.mla_debug_set_withhold(handle, 1)
        run(noalloc=True)
        assert lib.mla_decode_device_status(handle, None, stream) == mla.MLA_ERR_DEVICE_TIMEOUT
        lib.mla_debug_set_withhold(handle, 0)
        out.fill_(float("nan"))
        run(noalloc=True)   # each call copies the plan's header (zeroed counters) in first
        assert lib.mla_decode_device_status(handle, None, stream) == mla.MLA_OK
        assert torch.equal(out, clean_out) and torch.equal(lse, clean_lse)
    finally:
        lib.mla_plan_destroy(handle)
