"""Backward pass of one block on the F32 path against the gradient oracle.

Gate: every gradient (the block input's and the 12 weight gradients) at
max relative error <= 1e-4, the error measured as max_i |g - r| /
max(|r_i|, rms(r)) (the F32 gate of the forward).  fp32 accumulation over
the B T rows of a weight gradient (<= 1024 terms) and over the keys of a
softmax row errs by ~1e-6 relative; a dropped path (the variance term of the
LayerNorm gradient, the residual gradient, a softmax term) or a transposed
weight changes a gradient by O(1).
"""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_util import max_rel_err, rng, to_np, to_t

torch = pytest.importorskip("torch")
import gpt_pre_ln_gb300 as G  # noqa: E402

pytestmark = pytest.mark.gpu

KEYS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_fc", "b_fc", "w_proj", "b_proj")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gpt_pre_ln_gb300 import build
    build.build()
    G.lib()
    yield
    st, site = G.gpt2_last_error()
    assert st == 0, f"device error {st} at site {site}"


def _run(dims, layer, B, T, seed):
    params, d = synth.draw_model(dims, "f32", seed, with_embeddings=False)
    blk = params["blocks"][0]
    x = synth.draw_activations(d, B, T, dims.d_model)
    dy = synth.round_to(rng(seed + 1).standard_normal((B, T, dims.d_model)), "f32")
    flags = ((G.SCALE_ATTN_BY_INVERSE_LAYER_IDX if dims.scale_attn_by_inverse_layer_idx else 0)
             | (G.GELU_EXACT if dims.gelu_exact else 0))
    cd = G.make_dims(dims.n_layer, dims.d_model, dims.n_head, dims.d_ff, dims.vocab, dims.n_pos, dims.eps, G.F32,
                     flags=flags)
    dev = {k: to_t(v, "f32") for k, v in blk.items()}
    grads = {k: torch.full_like(dev[k], float("nan")) for k in KEYS}
    xt, dyt = to_t(x, "f32"), to_t(dy, "f32")
    dx = torch.full_like(xt, float("nan"))
    wsb = G.gpt2_block_backward_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_block_backward(cd, G.block_weights(dev), layer, xt, dyt, dx, G.block_grads(grads), B, T, ws, wsb)
    torch.cuda.synchronize()
    ref_dx, ref = O.block_backward(dy, x, blk, dims.n_head, dims.eps, layer, dims.scale_attn_by_inverse_layer_idx,
                                   dims.gelu_exact)
    return to_np(dx), {k: to_np(v) for k, v in grads.items()}, ref_dx, ref


@pytest.mark.parametrize("switches,layer", [((False, False), 0), ((True, True), 2)])
@pytest.mark.parametrize("B,T", [(2, 37), (1, 130)])
def test_block_backward_f32_small(switches, layer, B, T):
    dims = synth.Dims(n_layer=1, d_model=128, n_head=2, d_ff=320, vocab=1, n_pos=256,
                      scale_attn_by_inverse_layer_idx=switches[0], gelu_exact=switches[1])
    dx, g, ref_dx, ref = _run(dims, layer, B, T, 700 + T + layer)
    assert max_rel_err(dx, ref_dx) <= 1e-4
    for k in KEYS:
        assert max_rel_err(g[k], ref[k]) <= 1e-4, k


def test_block_backward_f32_gpt2_small_block():
    """A GPT-2 small block (D = 768, 12 heads, F = 3072), B = 1, T = 64."""
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=1)
    dx, g, ref_dx, ref = _run(dims, 0, 1, 64, 4242)
    assert max_rel_err(dx, ref_dx) <= 1e-4
    for k in KEYS:
        assert max_rel_err(g[k], ref[k]) <= 1e-4, k
    # the gradient reaches every weight
    for k in KEYS:
        assert np.abs(ref[k]).max() > 0


def test_block_backward_is_deterministic():
    dims = synth.Dims(n_layer=1, d_model=128, n_head=2, d_ff=512, vocab=1, n_pos=64)
    a = _run(dims, 0, 2, 40, 9)
    b = _run(dims, 0, 2, 40, 9)
    assert np.array_equal(a[0], b[0])
    for k in KEYS:
        assert np.array_equal(a[1][k], b[1][k]), k
