"""The whole-model training step on the tensor cores against the gradient oracle.

gpt2_forward_backward runs the bf16 forward keeping each block's
intermediates, the mean shifted cross-entropy, and the gradient of every
parameter (the products of every linear layer, of the tied lm_head and of
the causal attention backward on the tcgen05 tensor cores).  The oracle is
``loss_and_grads`` of the gradient oracle in float64 on the same bf16
weights and tokens.

Gates.  The loss: relative error <= 2e-3 (the forward's logits gate is a
rel L2 of 1e-2; the mean of lse - z over positions averages those errors).
Each gradient tensor: rel L2 <= 3e-2.  The bf16 path rounds every operand of
a product to 8 significant bits (2^-9 relative): the activations the forward
keeps, and in the backward each gradient that enters a product (dz, dx', dg,
du, dh, do, dqkv) and the attention's p and ds.  A gradient passes through
about six such roundings per block on its way from the loss, each adding an
independent ~2^-9 relative error, so a few times 2^-9 * sqrt(6 L) (about 1%
at 2-12 layers) is expected; 3e-2 sits above that and far below what a
wrong term gives (a dropped path or a transposed operand moves a tensor by
O(1)).
"""
import numpy as np
import pytest

import synth
from gpu_util import rel_l2, to_np
from oracle import gpt2_grad as OG

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


def _train_step(dims, params, tokens, flags=0):
    B, T = tokens.shape
    dev = G.to_device(params, G.BF16)
    mw, keep = G.model_weights(dev)
    cd = G.make_dims(dims.n_layer, dims.d_model, dims.n_head, dims.d_ff, dims.vocab, dims.n_pos, dims.eps, G.BF16,
                     flags)
    zeros = lambda a: torch.full(a.shape, float("nan"), device="cuda")  # noqa: E731 (every entry must be written)
    gd = {k: zeros(params[k]) for k in ("wte", "wpe", "lnf_g", "lnf_b")}
    gd["blocks"] = [{k: zeros(b[k]) for k in KEYS} for b in params["blocks"]]
    mg, keep_g = G.model_grads(gd)
    loss = torch.full((1,), float("nan"), device="cuda")
    wsb = G.gpt2_train_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    tok = torch.from_numpy(tokens).cuda()
    G.gpt2_forward_backward(cd, mw, tok, None, mg, loss, B, T, ws, wsb)
    torch.cuda.synchronize()
    del keep, keep_g
    return float(loss.item()), gd


def _compare(dims, params, tokens, gd, loss, flags=0, gate=3e-2):
    d = synth.replace_dims(dims, scale_attn_by_inverse_layer_idx=bool(flags & G.SCALE_ATTN_BY_INVERSE_LAYER_IDX),
                           gelu_exact=bool(flags & G.GELU_EXACT))
    ref_loss, ref = OG.loss_and_grads(tokens, tokens, params, d)
    assert abs(loss - ref_loss) <= 2e-3 * abs(ref_loss), (loss, ref_loss)
    errs = {}
    for k in ("wte", "wpe", "lnf_g", "lnf_b"):
        errs[k] = rel_l2(to_np(gd[k]), ref[k])
    for l, (gb, rb) in enumerate(zip(gd["blocks"], ref["blocks"])):
        for k in KEYS:
            errs[f"{l}.{k}"] = rel_l2(to_np(gb[k]), rb[k])
    worst = max(errs, key=errs.get)
    print(f"loss {loss:.6f} (oracle {ref_loss:.6f}); worst gradient rel L2 {errs[worst]:.3e} ({worst})")
    bad = {k: v for k, v in errs.items() if not v <= gate}
    assert not bad, bad
    return errs


def test_train_step_small_model():
    """Two layers, D = 128, 40 positions (the few-row loss path)."""
    dims = synth.Dims(n_layer=2, d_model=128, n_head=2, d_ff=512, vocab=1000, n_pos=64)
    params, d = synth.draw_model(dims, "bf16", 901)
    tokens = synth.draw_tokens(d, 2, 40, dims.vocab)
    loss, gd = _train_step(dims, params, tokens)
    _compare(dims, params, tokens, gd, loss)
    # rows of wpe past T carry no gradient
    assert torch.count_nonzero(gd["wpe"][40:]).item() == 0


def test_train_step_gpt2_small_width():
    """GPT-2 small width and vocabulary, two layers, B = 2, T = 256: the
    fused log-sum-exp lm_head, the CTA-pair GEMMs and several attention
    tiles."""
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2, n_pos=256)
    params, d = synth.draw_model(dims, "bf16", 902)
    tokens = synth.draw_tokens(d, 2, 256, dims.vocab)
    loss, gd = _train_step(dims, params, tokens)
    _compare(dims, params, tokens, gd, loss)


def test_train_step_switches_and_ragged():
    """The GPT2Config switches (layer-index attention scale, exact GELU),
    n_inner != 4D and a ragged T."""
    dims = synth.Dims(n_layer=3, d_model=128, n_head=2, d_ff=320, vocab=700, n_pos=200)
    params, d = synth.draw_model(dims, "bf16", 903)
    tokens = synth.draw_tokens(d, 3, 131, dims.vocab)
    flags = G.SCALE_ATTN_BY_INVERSE_LAYER_IDX | G.GELU_EXACT
    loss, gd = _train_step(dims, params, tokens, flags)
    _compare(dims, params, tokens, gd, loss, flags)


@pytest.mark.parametrize("d_model,n_head", [(1024, 16), (1600, 25)])
def test_train_step_wide_rows(d_model, n_head):
    """The GPT-2 medium and XL widths (the LayerNorm backward holds 8 and 13
    groups of four columns per lane), one layer, a ragged row count."""
    dims = synth.Dims(n_layer=1, d_model=d_model, n_head=n_head, d_ff=4 * d_model, vocab=600, n_pos=96)
    params, d = synth.draw_model(dims, "bf16", 905 + n_head)
    tokens = synth.draw_tokens(d, 3, 83, dims.vocab)
    loss, gd = _train_step(dims, params, tokens)
    _compare(dims, params, tokens, gd, loss)


def test_train_step_is_deterministic():
    dims = synth.Dims(n_layer=2, d_model=128, n_head=2, d_ff=512, vocab=1000, n_pos=300)
    params, d = synth.draw_model(dims, "bf16", 904)
    tokens = synth.draw_tokens(d, 2, 300, dims.vocab)
    l1, g1 = _train_step(dims, params, tokens)
    l2, g2 = _train_step(dims, params, tokens)
    assert l1 == l2
    assert torch.equal(g1["wte"], g2["wte"]) and torch.equal(g1["blocks"][0]["w_qkv"], g2["blocks"][0]["w_qkv"])


def test_train_step_gpt2_small_full_depth():
    """GPT-2 small (12 layers), one sequence of 1024 positions."""
    inp = synth.workload_inputs("gpt2_small_fwd_b8_t1024", B_override=1)
    dims, params, tokens = inp["dims"], inp["params"], inp["tokens"]
    loss, gd = _train_step(dims, params, tokens)
    _compare(dims, params, tokens, gd, loss)
