"""Pins of the oracle's decode prologue (RoPE on the rope dims, the cache write of the new
tokens, quantise-on-write), on CPU: closed forms of the rotation, its relative-position
property, the quantiser against an independent one (torch's float8 cast), and the slots
written."""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import (WORKLOADS, make_inputs, new_tokens, quantize_e4m3_per_token, quantize_int8_per_token,
                       rope_table)


def _inputs(lens, H=4, P=16, seed=90, fp8=False, int8=False, f16=False):
    return make_inputs(WORKLOADS["tiny"], kv_lens=list(lens), batch=len(lens), h_q=H, page_size=P, seed=seed,
                       fp8=fp8, int8=int8, f16=f16)


def _run(inp, qo_len, table, interleaved, seed=91):
    q_pe, ckv_new, kpe_new = new_tokens(inp, qo_len, seed)
    res = oracle.decode_prologue(q_pe, ckv_new, kpe_new, table, inp.kv_indices, inp.kv_indptr,
                                 inp.kv_last_page_len, qo_len, interleaved, inp.ckv, inp.kpe,
                                 ckv_scale=inp.ckv_scale)
    return (q_pe, ckv_new, kpe_new), res


def _slot(inp, b, t):
    P = inp.page_size
    return int(inp.kv_indices[int(inp.kv_indptr[b]) + t // P]), t % P


@pytest.mark.parametrize("interleaved", [True, False])
def test_position_zero_is_the_identity(interleaved):
    """cos 1, sin 0 at every position: the rotation leaves q_pe and kpe as they are."""
    inp = _inputs([1, 7, 40])
    table = torch.cat([torch.ones(64, 32), torch.zeros(64, 32)], dim=1)
    (q_pe, ckv_new, kpe_new), (q_out, ckv, kpe, _) = _run(inp, 1, table, interleaved)
    assert torch.equal(q_out, q_pe)
    for b, L in enumerate(inp.kv_lens.tolist()):
        pg, sl = _slot(inp, b, L - 1)
        assert torch.equal(kpe[pg, sl], kpe_new[b]) and torch.equal(ckv[pg, sl], ckv_new[b])


@pytest.mark.parametrize("interleaved", [True, False])
def test_quarter_turn_closed_form(interleaved):
    """cos 0, sin 1: every pair (a, b) becomes (-b, a), exactly; the pairing decides which dims move."""
    inp = _inputs([3, 20])
    table = torch.cat([torch.zeros(64, 32), torch.ones(64, 32)], dim=1)
    (q_pe, _, _), (q_out, _, _, _) = _run(inp, 1, table, interleaved)
    i = torch.arange(32)
    ia, ib = (2 * i, 2 * i + 1) if interleaved else (i, i + 32)
    assert torch.equal(q_out[..., ia], -q_pe[..., ib])
    assert torch.equal(q_out[..., ib], q_pe[..., ia])


@pytest.mark.parametrize("interleaved", [True, False])
def test_rotation_keeps_only_relative_position(interleaved):
    """<rope(q, t1), rope(k, t2)> depends on t1 - t2 alone, and the norm is kept."""
    table = rope_table(300)
    g = torch.Generator().manual_seed(5)
    q, k = torch.randn(64, generator=g, dtype=torch.float64), torch.randn(64, generator=g, dtype=torch.float64)
    rot = lambda x, t: oracle.rope_f64(x, table[t, :32], table[t, 32:], interleaved)
    for t1, t2, d in [(5, 3, 100), (40, 0, 7), (0, 90, 200)]:
        a = rot(q, t1) @ rot(k, t2)
        b = rot(q, t1 + d) @ rot(k, t2 + d)
        assert abs(a - b) <= 1e-5 * (1 + abs(a)), (a, b)   # the table is fp32
    assert abs(rot(q, 123).norm() - q.norm()) <= 1e-6 * q.norm()
    assert abs(rot(q, 0) @ rot(k, 0) - q @ k) <= 1e-12


def test_quantise_on_write_matches_the_cache_quantiser():
    """The 8-bit write equals quantize_e4m3_per_token (torch's float8 cast) on the same token:
    identical codes and scales; an all-zero token gets scale 0 and zero codes."""
    inp = _inputs([5, 33, 64, 100], fp8=True)
    q_pe, ckv_new, kpe_new = new_tokens(inp, 1, seed=92)
    ckv_new[2] = 0
    _, ckv, _, sc = oracle.decode_prologue(q_pe, ckv_new, kpe_new, rope_table(128), inp.kv_indices, inp.kv_indptr,
                                           inp.kv_last_page_len, 1, True, inp.ckv, inp.kpe, ckv_scale=inp.ckv_scale)
    codes, scale = quantize_e4m3_per_token(ckv_new.unsqueeze(1))
    for b, L in enumerate(inp.kv_lens.tolist()):
        pg, sl = _slot(inp, b, L - 1)
        assert torch.equal(ckv[pg, sl], codes[b, 0]), b
        assert sc[pg, sl].item() == scale[b, 0].item(), b
    pg, sl = _slot(inp, 2, 63)
    assert sc[pg, sl].item() == 0.0 and (ckv[pg, sl] == 0).all()


def test_int8_quantise_on_write_matches_the_cache_quantiser():
    """The INT8 write equals quantize_int8_per_token (torch's round-half-even) on the same token:
    identical codes and scales; an all-zero token gets scale 0 and zero codes."""
    inp = _inputs([5, 33, 64, 100], int8=True)
    q_pe, ckv_new, kpe_new = new_tokens(inp, 1, seed=93)
    ckv_new[1] = 0
    _, ckv, _, sc = oracle.decode_prologue(q_pe, ckv_new, kpe_new, rope_table(128), inp.kv_indices, inp.kv_indptr,
                                           inp.kv_last_page_len, 1, False, inp.ckv, inp.kpe, ckv_scale=inp.ckv_scale)
    codes, scale = quantize_int8_per_token(ckv_new.unsqueeze(1))
    for b, L in enumerate(inp.kv_lens.tolist()):
        pg, sl = _slot(inp, b, L - 1)
        assert torch.equal(ckv[pg, sl], codes[b, 0]), b
        assert sc[pg, sl].item() == scale[b, 0].item(), b
    pg, sl = _slot(inp, 1, 32)
    assert sc[pg, sl].item() == 0.0 and (ckv[pg, sl] == 0).all()


def test_f16_prologue_rounds_to_f16():
    """fp16 inputs: the rotation is rounded to fp16 (a quarter turn maps (a, b) to (-b, a)
    exactly, so the written kpe is exact), and the latent is copied bit for bit."""
    inp = _inputs([3, 40], f16=True)
    q_pe, ckv_new, kpe_new = new_tokens(inp, 1, seed=94, f16=True)
    table = torch.zeros(64, 64)
    table[:, 32:] = 1.0   # cos 0, sin 1 at every position: a quarter turn
    q_out, ckv, kpe, _ = oracle.decode_prologue(q_pe, ckv_new, kpe_new, table, inp.kv_indices, inp.kv_indptr,
                                                inp.kv_last_page_len, 1, False, inp.ckv, inp.kpe)
    assert q_out.dtype == torch.float16 and kpe.dtype == torch.float16
    for b, L in enumerate(inp.kv_lens.tolist()):
        pg, sl = _slot(inp, b, L - 1)
        a, bb = kpe_new[b, :32], kpe_new[b, 32:]
        assert torch.equal(kpe[pg, sl], torch.cat([-bb, a]))
        assert torch.equal(ckv[pg, sl].view(torch.int16), ckv_new[b].view(torch.int16))
    a, bb = q_pe[..., :32], q_pe[..., 32:]
    assert torch.equal(q_out, torch.cat([-bb, a], dim=-1))


@pytest.mark.parametrize("qo_len", [1, 3])
def test_only_the_new_tokens_slots_are_written(qo_len):
    """Rows b * qo_len + j write position L_b - qo_len + j; a request shorter than qo_len skips
    its missing positions; every other cache entry keeps its bits (NaN padding included)."""
    inp = _inputs([2, 17, 50], P=16)
    (q_pe, ckv_new, kpe_new), (q_out, ckv, kpe, _) = _run(inp, qo_len, rope_table(64), True)
    expect = {}
    for b, L in enumerate(inp.kv_lens.tolist()):
        for j in range(qo_len):
            t = L - qo_len + j
            if t >= 0:
                expect[_slot(inp, b, t)] = b * qo_len + j
            else:
                assert torch.equal(q_out[b * qo_len + j], q_pe[b * qo_len + j])   # untouched
    same_c = (ckv.view(torch.int16) == inp.ckv.view(torch.int16)).all(dim=-1)
    same_k = (kpe.view(torch.int16) == inp.kpe.view(torch.int16)).all(dim=-1)
    for pg in range(inp.ckv.shape[0]):
        for sl in range(inp.page_size):
            if (pg, sl) in expect:
                r = expect[(pg, sl)]
                assert torch.equal(ckv[pg, sl], ckv_new[r])
            else:
                assert same_c[pg, sl] and same_k[pg, sl], (pg, sl)
