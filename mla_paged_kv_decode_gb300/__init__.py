"""MLA paged-KV decode for one NVIDIA GB300 (sm_103a).

The computation runs in ``libmla_decode.so`` (hand-written CUDA: TMA page
staging, tcgen05/TMEM attention, deterministic split-KV combine); this package
is its ctypes binding.  ``Decoder`` bundles the usual call sequence
(plan -> workspace -> commit -> run) for callers that let torch own memory.
"""
from __future__ import annotations

from typing import Optional

import torch

from ._binding import (  # noqa: F401
    EXPORTED, MLA_ERR_CUDA, MLA_ERR_DEVICE_TIMEOUT, MLA_ERR_INVALID_ARG, MLA_ERR_NOT_COMMITTED,
    MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE_TOO_SMALL, MLA_KV_BF16, MLA_KV_FP8_E4M3, MLA_KV_INT8, MLA_KV_F16, MLA_OK, MLAError, Plan,
    library_path, load, mla_decode_device_status, mla_decode_plan, mla_decode_plan_commit,
    mla_decode_plan_workspace_bytes, mla_decode_run, mla_plan_get_segments, mla_plan_heads_per_cta,
    mla_plan_num_ctas, mla_plan_num_partials, mla_plan_num_segments, mla_status_string,
    mla_plan_num_launches, mla_decode_run_noalloc, mla_decode_noalloc_max_workspace_bytes,
    mla_plan_segment_cost_tiles, mla_plan_num_units, MLA_OUT_F32, MLA_OUT_BF16, mla_decode_plan_ex,
    mla_plan_num_rows, mla_decode_prologue,
)


def num_sms(device=None) -> int:
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


class Decoder:
    """Plan once for a batch composition, then run many times (graph-capturable).

    kv_indptr / kv_last_page_len are taken on the host for the plan and kept
    on the device for the kernels.  With qo_len > 1, q, out and lse hold
    batch * qo_len query rows (row b * qo_len + j is query token j of request b);
    out_dtype MLA_OUT_BF16 makes out bf16.
    """

    def __init__(self, kv_indptr: torch.Tensor, kv_last_page_len: torch.Tensor, h_q: int, page_size: int,
                 kv_dtype: int = MLA_KV_BF16, device=None, sms: Optional[int] = None, stream=None,
                 qo_len: int = 1, causal: bool = True, out_dtype: int = MLA_OUT_F32):
        device = torch.device(device or "cuda")
        self.batch = int(kv_indptr.numel()) - 1
        self.h_q, self.page_size, self.kv_dtype = h_q, page_size, kv_dtype
        self.qo_len, self.out_dtype = qo_len, out_dtype
        self.rows = self.batch * qo_len
        if qo_len == 1 and out_dtype == MLA_OUT_F32:
            self.plan = mla_decode_plan(kv_indptr.cpu(), kv_last_page_len.cpu(), self.batch, h_q, page_size,
                                        sms or num_sms(device), kv_dtype)
        else:
            self.plan = mla_decode_plan_ex(kv_indptr.cpu(), kv_last_page_len.cpu(), self.batch, qo_len, causal, h_q,
                                           page_size, sms or num_sms(device), kv_dtype, out_dtype)
        self.workspace = torch.empty(max(self.plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
        mla_decode_plan_commit(self.plan, self.workspace, stream)

    def run(self, q_nope, q_pe, ckv_cache, kpe_cache, kv_indices, kv_indptr, kv_last_page_len, sm_scale,
            ckv_scale=None, out=None, lse=None, stream=None):
        if out is None:
            odt = torch.bfloat16 if self.out_dtype == MLA_OUT_BF16 else torch.float32
            out = torch.empty(self.rows, self.h_q, 512, dtype=odt, device=q_nope.device)
        if lse is None:
            lse = torch.empty(self.rows, self.h_q, dtype=torch.float32, device=q_nope.device)
        mla_decode_run(self.plan, q_nope, q_pe, ckv_cache, ckv_scale, kpe_cache, kv_indices, kv_indptr,
                       kv_last_page_len, sm_scale, out, lse, self.workspace, stream)
        return out, lse

    def device_status(self, stream=None) -> int:
        return mla_decode_device_status(self.plan, self.workspace, stream)
