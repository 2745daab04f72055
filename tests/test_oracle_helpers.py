"""Pins for the two oracle helpers that every full-size parity test goes through.

``oracle.decode_inputs`` runs the oracle on a whole ``workloads.Inputs`` batch (or, for an
8-bit cache with ``use_bf16_cache``, on the bf16 cache it was quantised from), and
``oracle.decode_subset`` runs it on a subset of the batch's requests by slicing q and the
page table.  The oracle computes every request on its own with a fixed order of sums, so a
correct slice gives the whole batch's rows bit for bit; an independent restatement (the
torch brute force on the whole batch, then indexed) pins the same rows to 1e-12.

The FP8 acceptance test compares the GPU with the oracle on the original bf16 cache
(cosine <= 3e-3, FlashMLA PR #233, "Correctness": FP8 against bf16).  That check is only as
good as ``use_bf16_cache``: if the flag were ignored, the "bf16" reference would be the
dequantised one and the check vacuous.  ``test_planted_helper_mistakes_are_caught`` builds
copies of the helpers with such mistakes and checks that the pins here fail on each.
"""
import pytest
import torch

import oracle
from oracle.brute import brute_force
from workloads import WORKLOADS, make_inputs

# requests: empty, one token, one page exactly, several pages with a ragged last page
KV_LENS = (0, 1, 16, 37, 70, 0, 5, 129)
SUBSET = (6, 3, 0, 7, 1)   # out of order, with an empty request and a one-token one


def _ragged(fp8=False):
    return make_inputs(WORKLOADS["tiny"], kv_lens=list(KV_LENS), batch=len(KV_LENS), h_q=4, page_size=16,
                       pool_pages=40, seed=23, fp8=fp8)


def _same_bits(a, b):
    """Equal element for element, including -inf and the position of any NaN."""
    return a.shape == b.shape and torch.equal(torch.nan_to_num(a, nan=7.0, neginf=-9e300),
                                              torch.nan_to_num(b, nan=7.0, neginf=-9e300))


# ---------------------------------------------------------------- the pins, on any pair of helpers

def pin_subset_rows(decode_inputs, decode_subset, inp, use_bf16_cache=False):
    """decode_subset(inp, S)[i] == decode_inputs(inp)[S[i]] bit for bit."""
    full_o, full_l = decode_inputs(inp, use_bf16_cache=use_bf16_cache)
    sub_o, sub_l = decode_subset(inp, SUBSET, use_bf16_cache=use_bf16_cache)
    idx = torch.tensor(SUBSET)
    assert _same_bits(sub_o, full_o[idx]), "subset outputs differ from the whole batch's rows"
    assert _same_bits(sub_l, full_l[idx]), "subset lse differ from the whole batch's rows"


def pin_subset_brute(decode_subset, inp, use_bf16_cache=False):
    """decode_subset(inp, S) against the brute force on the whole batch, indexed by S."""
    if inp.ckv_scale is not None and not use_bf16_cache:
        ref_o, ref_l = brute_force(inp.q_nope, inp.q_pe, inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr,
                                   inp.kv_last_page_len, inp.sm_scale, ckv_scale=inp.ckv_scale)
    else:
        ckv = inp.ckv_bf16 if inp.ckv_scale is not None else inp.ckv
        ref_o, ref_l = brute_force(inp.q_nope, inp.q_pe, ckv, inp.kpe, inp.kv_indices, inp.kv_indptr,
                                   inp.kv_last_page_len, inp.sm_scale)
    sub_o, sub_l = decode_subset(inp, SUBSET, use_bf16_cache=use_bf16_cache)
    idx = torch.tensor(SUBSET)
    assert (sub_o - ref_o[idx]).abs().max().item() <= 1e-12
    fin = torch.isfinite(ref_l[idx])
    assert torch.equal(fin, torch.isfinite(sub_l))
    assert (sub_l[fin] - ref_l[idx][fin]).abs().max().item() <= 1e-12


def pin_bf16_cache_switch(decode_inputs, inp):
    """For an 8-bit workload, use_bf16_cache gives the oracle on inp.ckv_bf16 exactly, and
    differs from the result on the dequantised codes."""
    o16, l16 = decode_inputs(inp, use_bf16_cache=True)
    ref_o, ref_l = oracle.mla_decode(inp.q_nope, inp.q_pe, inp.ckv_bf16, inp.kpe, inp.kv_indices, inp.kv_indptr,
                                     inp.kv_last_page_len, inp.sm_scale)
    assert _same_bits(o16, ref_o) and _same_bits(l16, ref_l), "use_bf16_cache is not the bf16-cache oracle"
    o8, _ = decode_inputs(inp)
    fin = torch.isfinite(o8)
    # e4m3 keeps 3 mantissa bits: the dequantised cache moves every output visibly
    assert (o16[fin] - o8[fin]).abs().max().item() > 1e-3, "use_bf16_cache gives the dequantised result"


def pin_8bit_default(decode_inputs, inp):
    """Without the flag, an 8-bit workload runs on its codes and scales."""
    o8, l8 = decode_inputs(inp)
    ref_o, ref_l = oracle.mla_decode(inp.q_nope, inp.q_pe, inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr,
                                     inp.kv_last_page_len, inp.sm_scale, ckv_scale=inp.ckv_scale)
    assert _same_bits(o8, ref_o) and _same_bits(l8, ref_l)


def _all_pins(decode_inputs, decode_subset):
    bf16, fp8 = _ragged(), _ragged(fp8=True)
    return [
        lambda: pin_subset_rows(decode_inputs, decode_subset, bf16),
        lambda: pin_subset_rows(decode_inputs, decode_subset, fp8),
        lambda: pin_subset_rows(decode_inputs, decode_subset, fp8, use_bf16_cache=True),
        lambda: pin_subset_brute(decode_subset, bf16),
        lambda: pin_subset_brute(decode_subset, fp8),
        lambda: pin_subset_brute(decode_subset, fp8, use_bf16_cache=True),
        lambda: pin_bf16_cache_switch(decode_inputs, fp8),
        lambda: pin_8bit_default(decode_inputs, fp8),
    ]


# ---------------------------------------------------------------- the real helpers pass

def test_inputs_have_the_edge_cases():
    inp = _ragged()
    lens = [int(x) for x in inp.kv_lens]
    assert 0 in lens and 1 in lens and any(L > 2 * inp.page_size for L in lens)
    assert list(SUBSET) != sorted(SUBSET)


@pytest.mark.parametrize("k", range(8))
def test_helper_pins(k):
    _all_pins(oracle.decode_inputs, oracle.decode_subset)[k]()


# ---------------------------------------------------------------- planted mistakes are caught

def _plant_ignores_flag(inp, threads=0, use_bf16_cache=False):
    return oracle.decode_inputs(inp, threads=threads)


def _plant_subset_ignores_flag(inp, requests, threads=0, use_bf16_cache=False):
    return oracle.decode_subset(inp, requests, threads=threads)


def _plant_subset_unsliced_last(inp, requests, threads=0, use_bf16_cache=False):
    """Slices q and the page lists but keeps the first len(S) kv_last_page_len entries."""
    idx = torch.as_tensor(list(requests), dtype=torch.long)
    indptr = inp.kv_indptr.long()
    pieces = [inp.kv_indices[indptr[b]:indptr[b + 1]] for b in requests]
    sub_ptr = torch.zeros(len(pieces) + 1, dtype=torch.int32)
    sub_ptr[1:] = torch.cumsum(torch.tensor([len(p) for p in pieces]), 0).to(torch.int32)
    ckv, scale = (inp.ckv_bf16, None) if use_bf16_cache and inp.ckv_bf16 is not None else (inp.ckv, inp.ckv_scale)
    return oracle.mla_decode(inp.q_nope[idx], inp.q_pe[idx], ckv, inp.kpe, torch.cat(pieces), sub_ptr,
                             inp.kv_last_page_len[: len(requests)], inp.sm_scale, ckv_scale=scale, threads=threads)


def _plant_subset_sorted(inp, requests, threads=0, use_bf16_cache=False):
    """Returns the rows in ascending request order instead of the order asked for."""
    return oracle.decode_subset(inp, sorted(requests), threads=threads, use_bf16_cache=use_bf16_cache)


@pytest.mark.parametrize("plant", ["inputs_ignores_flag", "subset_ignores_flag", "subset_unsliced_last",
                                   "subset_sorted"])
def test_planted_helper_mistakes_are_caught(plant):
    di, ds = oracle.decode_inputs, oracle.decode_subset
    if plant == "inputs_ignores_flag":
        di = _plant_ignores_flag
    elif plant == "subset_ignores_flag":
        ds = _plant_subset_ignores_flag
    elif plant == "subset_unsliced_last":
        ds = _plant_subset_unsliced_last
    else:
        ds = _plant_subset_sorted
    failed = 0
    for pin in _all_pins(di, ds):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"planted helper mistake {plant} slipped past every pin"
