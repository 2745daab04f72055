"""The no-allocation entry point (mla_decode_run_noalloc) against the regular one.

Some callers cannot allocate device memory at all: their allocator must not be
re-entered from inside a decode step, or every device allocation belongs to a
framework or a memory pool fixed at start-up.  For them the library offers a
decode call that takes no workspace and uses a fixed device array inside the
library instead.  This test calls it twice in a row through the C ABI and checks
each result against mla_decode_run with a caller-allocated workspace, for three
plans whose long requests are split across CTAs (so the array holds partials and
merge counters): a 16-head bf16 cache (the narrow kernel), a 16-head e4m3 cache and
a 128-head bf16 cache (the two-CTA kernel, 256 KB per partial).  The same plan runs
the same kernel on the same inputs, so the results must agree bit for bit, between
the two entry points and between the two no-allocation calls.  The array's status
word is read back after each call (mla_decode_device_status with no workspace).

The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
from gpu_helpers import LSE_ABS, MAX_ABS, cos_dist
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

CASES = {
    # name: (kv_lens, h_q, page_size, fp8)
    "bf16_h16": ([3000, 1, 0, 700, 4096, 129], 16, 64, False),
    "e4m3_h16": ([3000, 1, 0, 700, 4096, 129], 16, 64, True),
    "bf16_h128": ([1500, 0, 300, 1], 128, 64, False),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_kv_decode_gb300 import build as lib_build
    if lib_build.needs_build():
        lib_build.build()
    mla.load()


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_workspace_path_twice(case):
    lib = mla.load()
    lens, H, P, fp8 = CASES[case]
    inp = make_inputs(WORKLOADS["tiny"], kv_lens=lens, batch=len(lens), h_q=H, page_size=P, seed=41, fp8=fp8)
    d = inp.to("cuda")
    kvd = mla.MLA_KV_FP8_E4M3 if fp8 else mla.MLA_KV_BF16
    plan = mla.mla_decode_plan(inp.kv_indptr, inp.kv_last_page_len, inp.batch, inp.h_q, inp.page_size,
                               mla.num_sms(), kv_dtype=kvd)
    assert mla.mla_plan_num_partials(plan) > 0          # split requests: partials and counters in the array
    assert plan.workspace_bytes <= lib.mla_decode_noalloc_max_workspace_bytes()

    # reference: caller-allocated workspace
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    mla.mla_decode_plan_commit(plan, ws)
    ref_out = torch.empty(inp.batch, inp.h_q, 512, device="cuda")
    ref_lse = torch.empty(inp.batch, inp.h_q, device="cuda")
    mla.mla_decode_run(plan, d.q_nope, d.q_pe, d.ckv, d.ckv_scale, d.kpe, d.kv_indices, d.kv_indptr,
                       d.kv_last_page_len, inp.sm_scale, ref_out, ref_lse, ws)
    torch.cuda.synchronize()
    assert mla.mla_decode_device_status(plan, ws) == mla.MLA_OK

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    results = []
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = lib.mla_decode_run_noalloc(plan.handle, ptr(d.q_nope), ptr(d.q_pe), ptr(d.ckv), ptr(d.ckv_scale),
                                        ptr(d.kpe), inp.num_pages, ptr(d.kv_indices), ptr(d.kv_indptr),
                                        ptr(d.kv_last_page_len), ctypes.c_float(inp.sm_scale), ptr(out), ptr(lse),
                                        stream)
        assert rc == mla.MLA_OK, mla.mla_status_string(rc)
        # the array's status word: no bounded wait ran out
        assert lib.mla_decode_device_status(plan.handle, None, stream) == mla.MLA_OK, f"call {call}"
        torch.cuda.synchronize()
        fin = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse), fin), f"call {call}: lse finiteness differs"
        assert (out - ref_out).abs().max().item() <= MAX_ABS, f"call {call}"
        assert cos_dist(out.cpu(), ref_out.cpu()) <= 1e-4, f"call {call}"
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= LSE_ABS, f"call {call}"
        # same plan, same kernel, same inputs: the same bits
        assert torch.equal(out, ref_out), f"call {call}: out differs from the workspace path"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from the workspace path"
        results.append((out, lse))
    assert torch.equal(results[0][0], results[1][0]) and torch.equal(results[0][1], results[1][1])


def test_noalloc_rejects_a_plan_larger_than_the_array():
    lib = mla.load()
    # 128 heads, many split requests: the partials alone exceed the fixed array
    lens = [32768] * 64
    P = 64
    n = [(L + P - 1) // P for L in lens]
    indptr = torch.tensor([0] + list(torch.cumsum(torch.tensor(n), 0)), dtype=torch.int32)
    last = torch.tensor([L - (k - 1) * P for L, k in zip(lens, n)], dtype=torch.int32)
    plan = mla.mla_decode_plan(indptr, last, len(lens), 128, P, 2048)
    assert plan.workspace_bytes > lib.mla_decode_noalloc_max_workspace_bytes()
    dummy = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = lib.mla_decode_run_noalloc(plan.handle, p, p, p, None, p, 1, p, p, p, ctypes.c_float(0.1), p, p, None)
    assert rc == mla.MLA_ERR_WORKSPACE_TOO_SMALL
