"""The decode layer (row f4) on the GPU against its fp64 oracle.

FlashMLA PR #233 ("What is added") builds the decode layer around the attention kernel: a
prologue kernel for RoPE and the cache write, the projections, and the whole layer as one
CUDA graph.  ``mla_paged_kv_decode_gb300.layer.DecodeLayer`` is that layer over this library
(cuBLAS GEMMs for the projections); ``oracle.layer.decode_layer`` computes the same steps in
fp64, rounding to bf16 where the layer stores a bf16 activation.

Bars: the layer's output y (bf16) within 2e-2 of the oracle's relative to max |y|, cosine
distance <= 1e-4 (the bf16 gates of the decode; a cuBLAS fp32 sum can round an intermediate
bf16 value the other way from the fp64 sum, and each such flip is one bf16 step); the new
tokens written into the cache within one bf16 step (the latent is rounded from a cuBLAS sum);
graph replay bit-identical to the eager step.  Full-size layer (DeepSeek-V2-Lite: 2048 wide,
16 heads), ragged cache lengths, page sizes 16 and 64, bf16 and e4m3 caches.
"""
import pytest
import torch

import mla_paged_kv_decode_gb300 as mla
from gpu_helpers import cos_dist
from mla_paged_kv_decode_gb300.layer import DecodeLayer, LayerWeights
from oracle.layer import decode_layer
from workloads import WORKLOADS, layer_hidden, layer_weights, make_inputs, rope_table

pytestmark = pytest.mark.gpu

ROPE = rope_table(8192)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_paged_kv_decode_gb300 import build as lib_build
    if lib_build.needs_build():
        lib_build.build()
    mla.load()


def _case(kv_lens, P, seed, fp8=False):
    inp = make_inputs(WORKLOADS["tiny"], kv_lens=list(kv_lens), batch=len(kv_lens), h_q=16, page_size=P, seed=seed,
                      fp8=fp8)
    w = layer_weights(seed + 1)
    x = layer_hidden(len(kv_lens), seed + 2)
    return inp, w, x


def _gpu_layer(inp, w, x, fp8):
    d = inp.to("cuda")
    kvd = mla.MLA_KV_FP8_E4M3 if fp8 else mla.MLA_KV_BF16
    layer = DecodeLayer(LayerWeights(**vars(w)).to("cuda"), inp.kv_indptr, inp.kv_last_page_len, inp.page_size,
                        ROPE, kv_dtype=kvd)
    return layer, d


@pytest.mark.parametrize("P", [16, 64])
@pytest.mark.parametrize("fp8", [False, True])
def test_layer_matches_oracle(P, fp8):
    inp, w, x = _case([1, 37, 300, 1025, 64], P, seed=200 + P, fp8=fp8)
    layer, d = _gpu_layer(inp, w, x, fp8)
    y = layer.step(x.cuda(), d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len, ckv_scale=d.ckv_scale)
    torch.cuda.synchronize()
    assert mla.mla_decode_device_status(layer.plan, layer.workspace) == mla.MLA_OK
    y_ref, ckv_ref, kpe_ref, sc_ref = decode_layer(x, w, inp.ckv, inp.kpe, inp.kv_indices, inp.kv_indptr,
                                                   inp.kv_last_page_len, ROPE, layer.sm_scale,
                                                   ckv_scale=inp.ckv_scale)
    y = y.cpu().double()
    assert torch.isfinite(y).all()
    scale = float(y_ref.abs().max())
    err = float((y - y_ref).abs().max())
    cd = cos_dist(y, y_ref)
    assert err <= 2e-2 * scale and cd <= 1e-4, f"max err {err:.3e} (max |y| {scale:.3f}) cos {cd:.2e}"
    # the new tokens' cache rows: kpe within one bf16 step; the latent likewise (bf16 cache) or
    # its codes within one e4m3 step and its scale within 1 % (e4m3 cache)
    P_ = inp.page_size
    for r, L in enumerate(inp.kv_lens.tolist()):
        page = int(inp.kv_indices[int(inp.kv_indptr[r]) + (L - 1) // P_])
        slot = (L - 1) % P_
        kg, kr = d.kpe[page, slot].cpu().double(), kpe_ref[page, slot].double()
        assert torch.allclose(kg, kr, rtol=2 ** -7, atol=1e-3), r
        if fp8:
            sg, sr = float(d.ckv_scale[page, slot]), float(sc_ref[page, slot])
            assert abs(sg - sr) <= 0.01 * abs(sr), (r, sg, sr)
            cg = d.ckv[page, slot].cpu().view(torch.float8_e4m3fn).double()
            cr = ckv_ref[page, slot].view(torch.float8_e4m3fn).double()
            assert float((cg - cr).abs().max()) <= 32.0 and float((cg != cr).double().mean()) <= 0.05, r
        else:
            cg, cr = d.ckv[page, slot].cpu().double(), ckv_ref[page, slot].double()
            assert torch.allclose(cg, cr, rtol=2 ** -7, atol=1e-3), r


def test_layer_graph_replay_is_bit_identical():
    inp, w, x = _case([900, 4096, 3, 2500], 64, seed=300)
    layer, d = _gpu_layer(inp, w, x, False)
    xd = x.cuda()
    y0 = layer.step(xd, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len).clone()
    y_static = layer.capture(xd, d.ckv, d.kpe, d.kv_indices, d.kv_indptr, d.kv_last_page_len)
    for _ in range(3):
        layer.replay()
        torch.cuda.synchronize()
        assert torch.equal(y_static, y0)
    assert mla.mla_decode_device_status(layer.plan, layer.workspace) == mla.MLA_OK
