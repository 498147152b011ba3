"""Pins for the float64 oracle: facts the pages and the mathematics fix.

Each test names the mistake it is there to catch.  Nothing here touches the
CUDA library; these run on any CPU.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle as O
import synth
from synth import Dims

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.Generator(np.random.PCG64(7))


def _blk(dims, seed=3, scale=1.0):
    params, _ = synth.draw_model(dims, "f32", seed, with_embeddings=False)
    b = {k: np.asarray(v, np.float64) for k, v in params["blocks"][0].items()}
    for k in ("w_qkv", "w_o", "w_fc", "w_proj"):
        b[k] = b[k] * scale
    return b


# ------------------------------------------------------------------ LayerNorm
def test_layer_norm_closed_form_unit_affine():
    """gamma=1, beta=0: each row has mean 0 and variance var/(var+eps).

    Catches: the unbiased (n-1) variance, eps outside the square root, eps
    dropped, a missing mean subtraction.  Rows are scaled so var ~ eps.
    """
    eps = 1e-5
    for D in (4, 768, 1600):
        x = RNG.standard_normal((16, D)) * np.logspace(-4, 1, 16)[:, None] + 3.0
        y = O.layer_norm(x, np.ones(D), np.zeros(D), eps)
        var = x.var(axis=-1)  # population variance
        assert np.allclose(y.mean(-1), 0.0, atol=1e-12)
        np.testing.assert_allclose(y.var(-1), var / (var + eps), rtol=1e-10)


def test_layer_norm_matches_torch_fp64():
    """Same result as torch's layer_norm in float64 with random gamma/beta."""
    x = RNG.standard_normal((33, 768)) * 2.0 + 0.5
    g = 1 + 0.1 * RNG.standard_normal(768)
    b = 0.1 * RNG.standard_normal(768)
    ref = Fn.layer_norm(torch.from_numpy(x), (768,), torch.from_numpy(g), torch.from_numpy(b), eps=1e-5).numpy()
    np.testing.assert_allclose(O.layer_norm(x, g, b, 1e-5), ref, rtol=1e-12, atol=1e-12)


def test_layer_norm_page_example_is_unpinned():
    """The worked LN example on the huaweicloud page (section 六) is garbled.

    Its outputs equal (x - mean) / 55.9, but 55.9 is neither the population
    (54.13) nor the sample (62.50) standard deviation of the input.  The test
    records that reading: the oracle's population std of the page's input
    is 54.13, and the page's printed outputs are not reproduced.
    """
    x = np.array([100.0, 0.001, -50.0, 25.0])
    assert abs(x.mean() - 18.75) < 1e-3
    assert abs(x.std() - 54.13) < 0.01
    y = O.layer_norm(x, np.ones(4), np.zeros(4), 1e-5)
    page = np.array([1.45, -0.34, -1.23, 0.11])
    assert np.max(np.abs(y - page)) > 0.05


# ------------------------------------------------------------------- gelu_new
def test_gelu_new_matches_torch_tanh_gelu():
    """Catches the erf GELU substituted for gelu_new, or a wrong constant."""
    x = np.linspace(-8, 8, 4001)
    ref = Fn.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(O.gelu_new(x), ref, rtol=1e-13, atol=1e-15)
    erf = Fn.gelu(torch.from_numpy(x)).numpy()
    assert np.max(np.abs(O.gelu_new(x) - erf)) > 1e-4


def test_gelu_new_special_values():
    assert O.gelu_new(0.0) == 0.0
    assert abs(O.gelu_new(20.0) - 20.0) < 1e-12
    assert abs(O.gelu_new(-20.0)) < 1e-12
    # a value computed by hand: x=1 -> 0.5*(1+tanh(sqrt(2/pi)*1.044715))
    assert abs(O.gelu_new(1.0) - 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * 1.044715))) < 1e-15


# ------------------------------------------------------------------ attention
def test_attention_probability_rows():
    """Rows sum to 1, future entries are exactly 0, row 0 is [1, 0, ...]."""
    q = RNG.standard_normal((2, 3, 37, 64))
    k = RNG.standard_normal((2, 3, 37, 64))
    p = O.causal_probs(q, k)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14)
    iu = np.triu_indices(37, 1)
    assert np.all(p[..., iu[0], iu[1]] == 0.0)
    assert np.all(p[..., 0, 0] == 1.0)


def test_attention_position0_and_identical_keys():
    """o_0 = v_0 exactly; identical keys give o_i = mean of v_0..v_i."""
    B, T, H, hd = 2, 29, 3, 64
    D = H * hd
    qkv = RNG.standard_normal((B, T, 3 * D))
    o = O.causal_attention(qkv, H)
    v = qkv[..., 2 * D:]
    np.testing.assert_array_equal(o[:, 0], v[:, 0])
    qkv2 = qkv.copy()
    qkv2[..., D:2 * D] = qkv2[:, :1, D:2 * D]  # every key equals key 0
    o2 = O.causal_attention(qkv2, H)
    cummean = np.cumsum(v, axis=1) / np.arange(1, T + 1)[None, :, None]
    np.testing.assert_allclose(o2, cummean, rtol=1e-12, atol=1e-13)


def test_attention_matches_torch_sdpa_fp64():
    """Catches a wrong scale, a mask off by one, Q/K/V or head columns mixed up.

    The head split here is written from the page's description with torch
    ops (split into Q|K|V along the last axis, view [B,T,H,hd], permute to
    [B,H,T,hd]) and attention is torch's causal SDPA (scale 1/sqrt(hd)).
    """
    B, T, H, hd = 2, 45, 4, 64
    D = H * hd
    qkv = RNG.standard_normal((B, T, 3 * D))
    t = torch.from_numpy(qkv)
    q, k, v = t.split(D, dim=2)
    sh = lambda z: z.view(B, T, H, hd).permute(0, 2, 1, 3)  # noqa: E731
    ref = Fn.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True)
    ref = ref.permute(0, 2, 1, 3).reshape(B, T, D).numpy()
    np.testing.assert_allclose(O.causal_attention(qkv, H), ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------- block
def test_block_zero_sublayers_is_identity():
    """All sublayer weights and biases zero: the block returns X exactly.

    "Hidden State 如何流过 GPT-2 Block", section Residual Connection: with the
    update F(x) = 0 the residual path alone gives x_new = x.
    """
    dims = Dims(1, 128, 2, 512, 11, 64)
    blk = _blk(dims)
    for k in ("w_qkv", "b_qkv", "w_o", "b_o", "w_fc", "b_fc", "w_proj", "b_proj"):
        blk[k] = np.zeros_like(blk[k])
    x = RNG.standard_normal((2, 17, 128))
    np.testing.assert_array_equal(O.block_forward(x, blk, 2, 1e-5), x)


def test_block_zero_weights_closed_form():
    """All four weight matrices zero, biases not: X' = X + b_o + b_proj.

    Q = K = V = b_qkv rows for every position, so attention returns b_v and
    c_proj maps it to b_o; the MLP returns b_proj.  Catches a dropped bias or
    a dropped residual in either sublayer.
    """
    dims = Dims(1, 128, 2, 512, 11, 64)
    blk = _blk(dims)
    for k in ("w_qkv", "w_o", "w_fc", "w_proj"):
        blk[k] = np.zeros_like(blk[k])
    x = RNG.standard_normal((3, 9, 128))
    np.testing.assert_allclose(O.block_forward(x, blk, 2, 1e-5), x + blk["b_o"] + blk["b_proj"],
                               rtol=0, atol=1e-14)


def test_block_shape_preserved():
    with open(os.path.join(GOLDEN, "shape_claims.json")) as f:
        g = json.load(f)["block_shapes"]
    for c in g["cases"]:
        D = c["D"]
        H = 2 if D == 4 else 12
        dims = Dims(1, D, H, 4 * D, 11, 64)
        x = RNG.standard_normal((c["B"], c["T"], D))
        assert O.block_forward(x, _blk(dims), H, 1e-5).shape == x.shape


# ------------------------------------------------------------ toy brute force
TOY = Dims(n_layer=2, d_model=4, n_head=2, d_ff=16, vocab=11, n_pos=3)


def _toy_params(dims, seed=11):
    p, d = synth.draw_model(dims, "f32", seed)
    # make LayerNorm affine and biases non-trivial so every term matters
    p = {k: (np.asarray(v, np.float64) if k != "blocks" else v) for k, v in p.items()}
    p["blocks"] = [{k: np.asarray(v, np.float64) * (10.0 if k.startswith("w_") else 1.0) for k, v in b.items()}
                   for b in p["blocks"]]
    for b in p["blocks"]:
        for k in ("b_qkv", "b_o", "b_fc", "b_proj", "ln1_b", "ln2_b"):
            b[k] = b[k] * 20
    p["wte"] = p["wte"] * 30
    p["wpe"] = p["wpe"] * 30
    return p


def _scalar_forward(tokens, p, dims):
    """An independent scalar expansion written with explicit loops.

    Indexing follows the pages directly: W[in][out], Q|K|V column blocks,
    head h owns columns h*hd .. h*hd+hd-1, key j visible to query i iff
    j <= i, scores divided by sqrt(hd), the lm_head dots with rows of wte.
    """
    D, H, F, V = dims.d_model, dims.n_head, dims.d_ff, dims.vocab
    hd = D // H
    T = len(tokens)

    def ln(v, g, b):
        mu = sum(v) / D
        var = sum((a - mu) ** 2 for a in v) / D
        return [g[i] * (v[i] - mu) / math.sqrt(var + dims.eps) + b[i] for i in range(D)]

    def lin(v, W, bias, n_in, n_out):
        return [bias[o] + sum(v[i] * W[i][o] for i in range(n_in)) for o in range(n_out)]

    def gelu(z):
        return 0.5 * z * (1 + math.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z * z * z)))

    xs = [[p["wte"][tokens[t]][i] + p["wpe"][t][i] for i in range(D)] for t in range(T)]
    for blk in p["blocks"]:
        qkv = [lin(ln(xs[t], blk["ln1_g"], blk["ln1_b"]), blk["w_qkv"], blk["b_qkv"], D, 3 * D) for t in range(T)]
        hs = []
        for i in range(T):
            o = [0.0] * D
            for h in range(H):
                qi = [qkv[i][h * hd + e] for e in range(hd)]
                sc = []
                for j in range(i + 1):
                    kj = [qkv[j][D + h * hd + e] for e in range(hd)]
                    sc.append(sum(qi[e] * kj[e] for e in range(hd)) / math.sqrt(hd))
                m = max(sc)
                ex = [math.exp(s - m) for s in sc]
                z = sum(ex)
                for e in range(hd):
                    o[h * hd + e] = sum(ex[j] / z * qkv[j][2 * D + h * hd + e] for j in range(i + 1))
            a = lin(o, blk["w_o"], blk["b_o"], D, D)
            hs.append([xs[i][c] + a[c] for c in range(D)])
        new = []
        for i in range(T):
            f = [gelu(z) for z in lin(ln(hs[i], blk["ln2_g"], blk["ln2_b"]), blk["w_fc"], blk["b_fc"], D, F)]
            m = lin(f, blk["w_proj"], blk["b_proj"], F, D)
            new.append([hs[i][c] + m[c] for c in range(D)])
        xs = new
    logits = []
    for i in range(T):
        y = ln(xs[i], p["lnf_g"], p["lnf_b"])
        logits.append([sum(y[c] * p["wte"][v][c] for c in range(D)) for v in range(V)])
    return np.array(logits)


@pytest.mark.parametrize("n_head", [1, 2])
def test_toy_stack_brute_force(n_head):
    """The pages' toy stack (d_model=4, 3 tokens, 2 layers) by brute force.

    "Transformer Stack" page, section 猫吃鱼: d_model=4, seq_len=3, two blocks,
    then LayerNorm and the output head; shapes (1,3,4) throughout.
    """
    import dataclasses
    dims = dataclasses.replace(TOY, n_head=n_head)
    p = _toy_params(dims)
    tokens = np.array([[3, 7, 1]])
    got = O.forward_logits(tokens, p, dims)
    assert got.shape == (1, 3, dims.vocab)
    ref = _scalar_forward(tokens[0], p, dims)
    np.testing.assert_allclose(got[0], ref, rtol=1e-11, atol=1e-11)
    assert O.forward_hidden(tokens, p, dims).shape == (1, 3, 4)


def _torch_model_logits(tokens, p, dims):
    """The stack as torch fp64 modules, from the pages' description.

    Pre-LN blocks (x + attn(ln_1(x)); x + mlp(ln_2(x))), Conv1D-style
    ``addmm(bias, x, W)``, tanh GELU, causal SDPA, learned positions, final
    LayerNorm and a head tied to wte.  The GPT2Config switches map onto
    SDPA's ``scale`` (1 / (sqrt(hd) (l + 1)) for layer l) and torch's exact
    GELU.
    """
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))  # noqa: E731
    D, H = dims.d_model, dims.n_head
    hd = D // H
    idx = torch.from_numpy(tokens)
    B, T = idx.shape
    x = t(p["wte"])[idx] + t(p["wpe"])[:T]
    for l, b in enumerate(p["blocks"]):
        a = Fn.layer_norm(x, (D,), t(b["ln1_g"]), t(b["ln1_b"]), eps=dims.eps)
        qkv = torch.addmm(t(b["b_qkv"]), a.reshape(-1, D), t(b["w_qkv"])).view(B, T, 3 * D)
        q, k, v = qkv.split(D, dim=2)
        sh = lambda z: z.view(B, T, H, hd).permute(0, 2, 1, 3)  # noqa: E731
        sc = 1.0 / math.sqrt(hd) / ((l + 1) if dims.scale_attn_by_inverse_layer_idx else 1)
        o = Fn.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True, scale=sc)
        o = o.permute(0, 2, 1, 3).reshape(B * T, D)
        x = x + torch.addmm(t(b["b_o"]), o, t(b["w_o"])).view(B, T, D)
        a = Fn.layer_norm(x, (D,), t(b["ln2_g"]), t(b["ln2_b"]), eps=dims.eps).reshape(-1, D)
        g = Fn.gelu(torch.addmm(t(b["b_fc"]), a, t(b["w_fc"])), approximate="none" if dims.gelu_exact else "tanh")
        x = x + torch.addmm(t(b["b_proj"]), g, t(b["w_proj"])).view(B, T, D)
    x = Fn.layer_norm(x, (D,), t(p["lnf_g"]), t(p["lnf_b"]), eps=dims.eps)
    return (x @ t(p["wte"]).T).numpy()


def test_small_stack_matches_torch_modules():
    dims = Dims(n_layer=3, d_model=128, n_head=2, d_ff=512, vocab=97, n_pos=40)
    p = _toy_params(dims, seed=5)
    for b in p["blocks"]:
        for k in ("w_qkv", "w_o", "w_fc", "w_proj"):
            b[k] = b[k] / 10.0
    tokens = RNG.integers(0, dims.vocab, size=(2, 37)).astype(np.int32)
    np.testing.assert_allclose(O.forward_logits(tokens, p, dims), _torch_model_logits(tokens, p, dims),
                               rtol=1e-10, atol=1e-10)


# ------------------------------------------------------------------ causality
def test_causality_future_tokens_do_not_change_past_logits():
    """Changing tokens after position i leaves logits 0..i bit-identical."""
    dims = Dims(n_layer=2, d_model=128, n_head=2, d_ff=512, vocab=50, n_pos=32)
    p = _toy_params(dims, seed=9)
    tokens = RNG.integers(0, dims.vocab, size=(1, 32)).astype(np.int32)
    base = O.forward_logits(tokens, p, dims)
    for i in (0, 7, 30):
        t2 = tokens.copy()
        t2[0, i + 1:] = (t2[0, i + 1:] + 13) % dims.vocab
        got = O.forward_logits(t2, p, dims)
        assert np.array_equal(got[0, :i + 1], base[0, :i + 1])
        if i + 1 < 32:
            assert not np.allclose(got[0, i + 1:], base[0, i + 1:])


# --------------------------------------------------------- parameter layout
def test_gpt2_small_parameter_table():
    """Generator shapes reproduce the page's GPT-2 small parameter table."""
    with open(os.path.join(GOLDEN, "gpt2_small_param_table.json")) as f:
        g = json.load(f)
    dims = synth.GPT2_SMALL
    s = synth.param_shapes(dims)
    prod = lambda sh: int(np.prod(sh))  # noqa: E731
    blk = s["block"]
    counts = {
        "wte": prod(s["wte"]),
        "wpe": prod(s["wpe"]),
        "attention": dims.n_layer * sum(prod(blk[k]) for k in ("w_qkv", "b_qkv", "w_o", "b_o")),
        "ffn": dims.n_layer * sum(prod(blk[k]) for k in ("w_fc", "b_fc", "w_proj", "b_proj")),
        "layernorm": dims.n_layer * sum(prod(blk[k]) for k in ("ln1_g", "ln1_b", "ln2_g", "ln2_b"))
        + prod(s["lnf_g"]) + prod(s["lnf_b"]),
    }
    for k in ("wte", "wpe", "attention", "ffn", "layernorm"):
        assert counts[k] == g[k], k
    assert sum(counts.values()) == 124_439_808
    assert len(blk) == 12


def test_toy_param_count_matches_draw():
    p, _ = synth.draw_model(TOY, "f32", 1)
    c = synth.param_count(p)
    s = synth.param_shapes(TOY)
    assert c["wte"] == int(np.prod(s["wte"]))
    assert len(p["blocks"]) == 2 and len(p["blocks"][0]) == 12


def test_logits_shape_claim():
    """[1, 3] token ids give [1, 3, V] logits (page: torch.Size([1, 3, 50257]))."""
    with open(os.path.join(GOLDEN, "shape_claims.json")) as f:
        g = json.load(f)["logits_shape"]
    dims = Dims(n_layer=1, d_model=64, n_head=1, d_ff=256, vocab=g["vocab"], n_pos=8)
    p, _ = synth.draw_model(dims, "f32", 2)
    out = O.forward_logits(np.array(g["tokens"]), p, dims)
    assert list(out.shape) == g["expected"]


# --------------------------------------------------------------------- decode
def test_decode_step_equals_full_forward_row():
    """A decode step at position p equals row p of a full forward.

    "逐行拆GPT-2源码": with past_key_values the positions continue at
    past_length and the new K, V are concatenated after the cached ones.
    """
    dims = Dims(n_layer=2, d_model=128, n_head=2, d_ff=512, vocab=61, n_pos=24)
    p = _toy_params(dims, seed=4)
    tokens = RNG.integers(0, dims.vocab, size=(3, 20)).astype(np.int32)
    full = O.forward_logits(tokens, p, dims)
    P = 15
    cache = O.prefill_cache(tokens[:, :P], p, dims, T_max=24)
    past = np.full(3, P, np.int32)
    for step in range(P, 20):
        nxt, logits, cache, past = O.decode_step(p, dims, cache, past, tokens[:, step])
        np.testing.assert_allclose(logits, full[:, step], rtol=1e-10, atol=1e-10)
        np.testing.assert_array_equal(nxt, np.argmax(full[:, step], -1))
    assert np.all(past == 20)


def test_decode_ragged_past_lengths():
    """Sequences at different positions decode independently."""
    dims = Dims(n_layer=1, d_model=128, n_head=2, d_ff=512, vocab=33, n_pos=16)
    p = _toy_params(dims, seed=8)
    tokens = RNG.integers(0, dims.vocab, size=(2, 12)).astype(np.int32)
    full = O.forward_logits(tokens, p, dims)
    cache = np.zeros((1, 2, 2, 2, 16, 64))
    for b, P in ((0, 5), (1, 11)):
        cache[:, :, b:b + 1] = O.prefill_cache(tokens[b:b + 1, :P], p, dims, T_max=16)
    _, logits, _, _ = O.decode_step(p, dims, cache, np.array([5, 11]), np.array([tokens[0, 5], tokens[1, 11]]))
    np.testing.assert_allclose(logits[0], full[0, 5], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(logits[1], full[1, 11], rtol=1e-10, atol=1e-10)


def test_argmax_ties_lowest_index():
    assert O.argmax_lowest(np.array([[1.0, 3.0, 3.0, 2.0]]))[0] == 1


# ------------------------------------------------------------ synth rounding
def test_bf16_rounding_matches_torch():
    x = RNG.standard_normal(100000) * np.logspace(-3, 3, 100000)
    ours = synth.round_to(x, "bf16")
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_embed_positions_continue_at_offset():
    """Positions start at past_length: embedding a suffix at offset p equals
    the suffix of the embedding of the whole sequence ("逐行拆GPT-2源码",
    GPT2Model: position_ids = arange(past_length, past_length + T))."""
    wte = RNG.standard_normal((50, 8))
    wpe = RNG.standard_normal((20, 8))
    tokens = RNG.integers(0, 50, size=(2, 20))
    full = O.embed(tokens, wte, wpe)
    for p in (1, 7, 19):
        np.testing.assert_array_equal(O.embed(tokens[:, p:], wte, wpe, pos0=p), full[:, p:])


# ------------------------------------------------------------------ loss
def test_loss_uniform_logits_is_log_vocab():
    """All logits equal: every position's loss and lse are ln V exactly.

    Catches: a missing log, a sum where a mean belongs, lse without the
    maximum added back.
    """
    for V in (3, 50257):
        z = np.full((2, 5, V), 0.37)
        lab = RNG.integers(0, V, size=(2, 5))
        tl, lse, mean = O.shifted_cross_entropy(z, lab)
        np.testing.assert_allclose(tl, math.log(V), rtol=1e-14)
        np.testing.assert_allclose(lse, 0.37 + math.log(V), rtol=1e-14)
        assert tl.shape == (2, 4) and lse.shape == (2, 5)
        assert abs(mean - math.log(V)) < 1e-12


def test_loss_one_hot_margin_closed_form():
    """Target logit L above V-1 others at 0: loss = ln(1 + (V-1) e^-L).

    Catches: the sign of the target term, the target taken from the wrong
    column, overflow without the max shift (L = 800).
    """
    V = 11
    for L in (0.0, 2.5, 30.0, 800.0):
        z = np.zeros((1, 2, V))
        lab = np.array([[4, 7]])
        z[0, 0, 7] = L
        tl, lse, _ = O.shifted_cross_entropy(z, lab)
        assert np.isfinite(lse).all()
        # lse - L cancels: the absolute error is a few ulp of L
        np.testing.assert_allclose(tl[0, 0], math.log1p((V - 1) * math.exp(-L)), rtol=1e-12, atol=8 * np.spacing(max(L, 1.0)))


def test_loss_shift_uses_next_label():
    """Position t is scored against labels[t + 1]; labels[0] never counts.

    Catches: an unshifted loss, a shift the wrong way, scoring the last
    position.
    """
    V, T = 13, 6
    z = RNG.standard_normal((2, T, V)) * 3
    lab = RNG.integers(0, V, size=(2, T))
    tl, _, m0 = O.shifted_cross_entropy(z, lab)
    lab2 = lab.copy()
    lab2[:, 0] = (lab[:, 0] + 5) % V
    assert np.array_equal(O.shifted_cross_entropy(z, lab2)[0], tl)
    lab3 = lab.copy()
    lab3[1, 3] = (lab[1, 3] + 1) % V
    tl3 = O.shifted_cross_entropy(z, lab3)[0]
    changed = np.argwhere(tl3 != tl)
    assert changed.tolist() == [[1, 2]]
    z2 = z.copy()
    z2[:, -1] += 100.0  # the last position's logits are not scored
    assert O.shifted_cross_entropy(z2, lab)[2] == m0


def test_loss_matches_torch_cross_entropy_fp64():
    """The shifted mean equals torch's cross_entropy on the shifted tensors
    (float64), and lse equals torch.logsumexp."""
    V, B, T = 50, 3, 7
    z = RNG.standard_normal((B, T, V)) * 4
    lab = RNG.integers(0, V, size=(B, T))
    tl, lse, mean = O.shifted_cross_entropy(z, lab)
    zt = torch.from_numpy(z)
    ref = Fn.cross_entropy(zt[:, :-1].reshape(-1, V), torch.from_numpy(lab[:, 1:]).reshape(-1), reduction="none")
    np.testing.assert_allclose(tl.reshape(-1), ref.numpy(), rtol=1e-13)
    np.testing.assert_allclose(mean, ref.mean().item(), rtol=1e-13)
    np.testing.assert_allclose(lse, torch.logsumexp(zt, -1).numpy(), rtol=1e-13)


def test_loss_row_shift_invariance():
    """Adding c to every logit of a row leaves its loss unchanged and moves
    its lse by c (softmax is shift-invariant)."""
    V = 17
    z = RNG.standard_normal((1, 4, V))
    lab = RNG.integers(0, V, size=(1, 4))
    tl, lse, _ = O.shifted_cross_entropy(z, lab)
    c = np.array([5.0, -3.0, 40.0, 0.25])[None, :, None]
    tl2, lse2, _ = O.shifted_cross_entropy(z + c, lab)
    np.testing.assert_allclose(tl2, tl, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse + c[..., 0], rtol=1e-13)


def test_forward_loss_zero_wte_is_log_vocab():
    """wte = 0 makes every logit 0 whatever the blocks compute (the head is
    tied to wte): the loss is ln V at every position."""
    dims = Dims(n_layer=2, d_model=8, n_head=2, d_ff=32, vocab=19, n_pos=6, eps=1e-5)
    params, d = synth.draw_model(dims, "f32", 5)
    params["wte"] = np.zeros_like(params["wte"])
    tok = RNG.integers(0, dims.vocab, size=(2, 6))
    tl, lse, mean = O.forward_loss(tok, tok, params, dims)
    np.testing.assert_allclose(tl, math.log(19), rtol=1e-14)
    assert abs(mean - math.log(19)) < 1e-13


def test_loss_rejects_bad_labels():
    z = np.zeros((1, 3, 5))
    with pytest.raises(ValueError):
        O.shifted_cross_entropy(z, np.array([[0, 5, 1]]))
    with pytest.raises(ValueError):
        O.shifted_cross_entropy(np.zeros((1, 1, 5)), np.array([[0]]))


def test_prefill_cache_equals_token_by_token_decode():
    """The cache of a forward over T positions equals the cache that T decode
    steps from an empty cache build one token at a time ("逐行拆GPT-2源码":
    `present` is the concatenation of every step's K and V).

    Catches: K and V swapped, a head or position transposed, the cache of
    the wrong layer.
    """
    dims = Dims(n_layer=2, d_model=128, n_head=2, d_ff=512, vocab=29, n_pos=12)
    p = _toy_params(dims, seed=6)
    tokens = RNG.integers(0, dims.vocab, size=(2, 9)).astype(np.int32)
    ref = O.prefill_cache(tokens, p, dims, T_max=12)
    cache = np.zeros_like(ref)
    past = np.zeros(2, np.int32)
    for t in range(9):
        _, _, cache, past = O.decode_step(p, dims, cache, past, tokens[:, t])
    np.testing.assert_allclose(cache, ref, rtol=1e-11, atol=1e-12)
    assert np.all(ref[:, :, :, :, 9:] == 0)


# ------------------------------------------------ GPT2Config variants
def test_gelu_exact_matches_torch_and_identities():
    """x Phi(x): torch's exact GELU in fp64; Phi(1) = 0.8413447460685429;
    gelu(-x) = gelu(x) - x (Phi(-x) = 1 - Phi(x)); the tanh form of the
    pages stays within 1e-3 of it.

    Catches: a missing 1/sqrt(2), the tanh form in place of erf, a sign.
    """
    x = np.linspace(-8, 8, 4001)
    ref = Fn.gelu(torch.from_numpy(x), approximate="none").numpy()
    np.testing.assert_allclose(O.gelu_exact(x), ref, rtol=1e-13, atol=1e-15)
    assert abs(O.gelu_exact(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15
    np.testing.assert_allclose(O.gelu_exact(-x), O.gelu_exact(x) - x, rtol=1e-12, atol=1e-13)
    assert np.max(np.abs(O.gelu_exact(x) - O.gelu_new(x))) < 1e-3
    assert np.max(np.abs(O.gelu_exact(x) - O.gelu_new(x))) > 1e-5  # the two differ


def test_attention_extra_scale_matches_sdpa_and_scales_q():
    """With scale_attn_by_inverse_layer_idx, layer l's scores are divided by
    l + 1 as well: torch SDPA with scale 1/(8 (l + 1)) in fp64, and the same
    as attention with every query divided by l + 1."""
    B, T, H = 2, 33, 2
    qkv = RNG.standard_normal((B, T, 3 * 64 * H)) * 2.0
    for l in (0, 1, 5):
        got = O.causal_attention(qkv, H, O.attn_extra_scale(l, True))
        q, k, v = (torch.from_numpy(z) for z in O.split_qkv_heads(qkv, H))
        ref = Fn.scaled_dot_product_attention(q, k, v, is_causal=True, scale=1.0 / (8.0 * (l + 1)))
        np.testing.assert_allclose(got, O.merge_heads(ref.numpy()), rtol=1e-12, atol=1e-13)
        qkv2 = qkv.copy()
        qkv2[..., :64 * H] /= (l + 1)
        np.testing.assert_allclose(got, O.causal_attention(qkv2, H), rtol=1e-12, atol=1e-13)
    assert O.attn_extra_scale(3, False) == 1.0


def test_variant_stack_matches_torch_modules():
    """Both switches on and n_inner = 192 (not 4 D = 512): the oracle against
    the torch module stack.  The weights are large enough that the switches
    change the logits by far more than the tolerance (checked), so a switch
    the oracle ignored would fail."""
    base = Dims(n_layer=3, d_model=128, n_head=2, d_ff=192, vocab=61, n_pos=40)
    var = Dims(n_layer=3, d_model=128, n_head=2, d_ff=192, vocab=61, n_pos=40,
               scale_attn_by_inverse_layer_idx=True, gelu_exact=True)
    p = _toy_params(base, seed=9)
    for b in p["blocks"]:
        for k in ("w_qkv", "w_o", "w_fc", "w_proj"):
            b[k] = b[k] / 2.0
    assert p["blocks"][0]["w_fc"].shape == (128, 192)
    tokens = RNG.integers(0, base.vocab, size=(2, 29)).astype(np.int32)
    got = O.forward_logits(tokens, p, var)
    np.testing.assert_allclose(got, _torch_model_logits(tokens, p, var), rtol=1e-10, atol=1e-10)
    assert np.max(np.abs(got - O.forward_logits(tokens, p, base))) > 1e-4
    for one in (Dims(**{**base.__dict__, "gelu_exact": True}),
                Dims(**{**base.__dict__, "scale_attn_by_inverse_layer_idx": True})):
        np.testing.assert_allclose(O.forward_logits(tokens, p, one), _torch_model_logits(tokens, p, one),
                                   rtol=1e-10, atol=1e-10)


def test_inverse_layer_scale_leaves_layer_zero():
    """Layer 0 is divided by 1: a one-layer model is the same with the
    switch on or off."""
    d0 = Dims(n_layer=1, d_model=128, n_head=2, d_ff=512, vocab=31, n_pos=20)
    d1 = Dims(n_layer=1, d_model=128, n_head=2, d_ff=512, vocab=31, n_pos=20, scale_attn_by_inverse_layer_idx=True)
    p = _toy_params(d0, seed=2)
    tokens = RNG.integers(0, 31, size=(1, 17)).astype(np.int32)
    assert np.array_equal(O.forward_logits(tokens, p, d0), O.forward_logits(tokens, p, d1))


def test_variant_decode_and_prefill_follow_the_switches():
    """Decode after prefill equals the full forward's rows with both
    switches on (the decode path takes the layer-indexed scale and the exact
    GELU too)."""
    dims = Dims(n_layer=2, d_model=128, n_head=2, d_ff=192, vocab=41, n_pos=24,
                scale_attn_by_inverse_layer_idx=True, gelu_exact=True)
    p = _toy_params(dims, seed=12)
    tokens = RNG.integers(0, dims.vocab, size=(2, 16)).astype(np.int32)
    full = O.forward_logits(tokens, p, dims)
    cache = O.prefill_cache(tokens[:, :10], p, dims, T_max=24)
    past = np.full(2, 10, np.int32)
    for step in range(10, 16):
        _, logits, cache, past = O.decode_step(p, dims, cache, past, tokens[:, step])
        np.testing.assert_allclose(logits, full[:, step], rtol=1e-10, atol=1e-10)
