"""Pins of the decode-layer oracle (oracle/layer.py), on CPU.

The layer composes pinned parts (the decode oracle, the prologue restatement) with plain
fp64 matmuls; what needs pinning is the wiring: which projection feeds which input, the head
order, the new token's cache write, and the rotated q_pe.  Each pin is a closed form the
layer reduces to in a special case (FlashMLA PR #233, "What is added": the fused decode layer;
"Benchmarking MLA": the absorbed form, K = ckv ‖ kpe, V = ckv):

* one token per request: attention returns that token's latent, so y = ((x W_kv) W_UV) W_o;
* W_q = 0: every score is 0, attention is the mean of the cached latents;
* a constructed W_q, W_UK that make head h's query a large multiple of cached token t_h's
  latent: attention returns ckv_{t_h} for head h;
* q_pe rows equal to k_pe (W_q's rope part = W_kpe), scaled up: the new token's rotated key
  matches each rotated query exactly, so attention returns the new token's latent (an old
  token holding the unrotated k_pe would win instead if the query were not rotated).

Every planted mistake of ``oracle.layer.PLANTS`` fails at least one pin.
"""

import numpy as np
import pytest
import torch

from oracle.layer import PLANTS, decode_layer
from workloads import WORKLOADS, layer_hidden, layer_weights, make_inputs, rope_table

D, H, DN, DV = 128, 16, 32, 32   # a small layer: the attention sizes (512, 64) are the method's
SM_SCALE = (DN + 64) ** -0.5
ROPE = rope_table(4096)


def _bf(t):
    return t.to(torch.float64).to(torch.bfloat16).to(torch.float64)


def _inputs(kv_lens, P, seed):
    return make_inputs(WORKLOADS["tiny"], kv_lens=list(kv_lens), batch=len(kv_lens), h_q=H, page_size=P, seed=seed)


def _run(inp, w, x, plant=""):
    return decode_layer(x, w, inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr, inp.kv_last_page_len, ROPE, SM_SCALE,
                        plant=plant)


def _tail(o_lat, w):
    """y from the attention output o_lat [B, H, 512] (fp64 holding bf16 values), head by head."""
    B = o_lat.shape[0]
    o = torch.zeros(B, H, DV, dtype=torch.float64)
    for h in range(H):
        o[:, h] = _bf(o_lat[:, h] @ w.w_uv[h].to(torch.float64))
    return _bf(o.reshape(B, H * DV) @ w.w_o.to(torch.float64))


def _tokens(inp, b, ckv):
    """Request b's cached latents [L, 512] (fp64), in token order."""
    P = ckv.shape[1]
    n0, n1 = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
    L = (n1 - n0 - 1) * P + int(inp.kv_last_page_len[b])
    return torch.stack([ckv[int(inp.kv_indices[n0 + t // P]), t % P].to(torch.float64) for t in range(L)])


def _close(a, b):
    return torch.allclose(a, b, rtol=2 ** -7, atol=1e-6)


def pin_single_token(plant=""):
    inp = _inputs([1, 1, 1], 16, seed=1)
    w = layer_weights(11, D, H, DN, DV)
    x = layer_hidden(3, 12, D)
    y, ckv2, _, _ = _run(inp, w, x, plant)
    c = _bf(x.to(torch.float64) @ w.w_kv.to(torch.float64))
    return _close(y, _tail(c.unsqueeze(1).expand(3, H, 512), w))


def pin_uniform(plant=""):
    inp = _inputs([5, 40, 17], 16, seed=2)
    w = layer_weights(21, D, H, DN, DV)
    w.w_q = torch.zeros_like(w.w_q)
    x = layer_hidden(3, 22, D)
    y, ckv2, _, _ = _run(inp, w, x, plant)
    c = _bf(x.to(torch.float64) @ w.w_kv.to(torch.float64))
    means = []
    for b in range(3):
        toks = _tokens(inp, b, inp.ckv)
        toks[-1] = c[b]   # the new token, written by the prologue
        means.append(_bf(toks.mean(0)))
    return _close(y, _tail(torch.stack(means).unsqueeze(1).expand(3, H, 512), w))


def pin_dominant_token(plant=""):
    inp = _inputs([40], 16, seed=3)
    w = layer_weights(31, D, H, DN, DV)
    x = layer_hidden(1, 32, D)
    xf = x[0].to(torch.float64)
    toks = _tokens(inp, 0, inp.ckv)          # cached latents (the last slot becomes the new token)
    targets = [(3 * h + 1) % 39 for h in range(H)]   # distinct old tokens, one per head
    w_q = torch.zeros(D, H, DN + 64, dtype=torch.float64)
    w_uk = torch.zeros(H, DN, 512, dtype=torch.float64)
    for h in range(H):
        w_q[:, h, 0] = 2.0 * xf / (xf @ xf)   # q_nope[h] = ~2 e_0, q_pe = 0
        w_uk[h, 0] = toks[targets[h]]         # q_abs[h] = ~2 ckv_{t_h}
    w.w_q, w.w_uk = w_q.to(torch.bfloat16), w_uk.to(torch.bfloat16)
    y, _, _, _ = _run(inp, w, x, plant)
    o_lat = torch.stack([toks[targets[h]] for h in range(H)]).unsqueeze(0)
    return _close(y, _tail(o_lat, w))


def pin_rope_self_match(plant=""):
    inp = _inputs([50, 23], 16, seed=4)
    w = layer_weights(41, D, H, DN, DV)
    w.w_kpe = (w.w_kpe.to(torch.float32) * 12.0).to(torch.bfloat16)   # |k_pe| ~ 100
    w_q = torch.zeros(D, H, DN + 64, dtype=torch.bfloat16)
    w_q[:, :, DN:] = w.w_kpe.unsqueeze(1)    # q_pe[h] = k_pe for every head, q_nope = 0
    w.w_q = w_q
    x = layer_hidden(2, 42, D)
    # request b's first cached token gets kpe = k_b unrotated: a query left unrotated would match
    # it exactly and pick that token instead of the new one
    k = _bf(x.to(torch.float64) @ w.w_kpe.to(torch.float64)).to(torch.bfloat16)
    for b in range(2):
        inp.kpe[int(inp.kv_indices[int(inp.kv_indptr[b])]), 0] = k[b]
    y, _, _, _ = _run(inp, w, x, plant)
    c = _bf(x.to(torch.float64) @ w.w_kv.to(torch.float64))
    return _close(y, _tail(c.unsqueeze(1).expand(2, H, 512), w))


PINS = [pin_single_token, pin_uniform, pin_dominant_token, pin_rope_self_match]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_layer_pin(pin):
    assert pin()


@pytest.mark.parametrize("plant", PLANTS)
def test_each_planted_mistake_fails_a_pin(plant):
    failed = [p.__name__ for p in PINS if not p(plant)]
    assert failed, f"planted mistake {plant!r} passes every pin"


def test_layer_writes_the_new_token_only():
    """The prologue step of the layer changes exactly the new tokens' slots."""
    inp = _inputs([5, 40, 17], 16, seed=5)
    w = layer_weights(51, D, H, DN, DV)
    x = layer_hidden(3, 52, D)
    _, ckv2, kpe2, _ = _run(inp, w, x)
    a, b = inp.ckv.view(torch.int16).numpy(), ckv2.view(torch.int16).numpy()
    changed = np.argwhere((a != b).any(axis=2))
    P = inp.page_size
    want = set()
    for r in range(3):
        L = int(inp.kv_lens[r])
        want.add((int(inp.kv_indices[int(inp.kv_indptr[r]) + (L - 1) // P]), (L - 1) % P))
    assert {tuple(map(int, c)) for c in changed} == want
