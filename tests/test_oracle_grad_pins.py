"""Pins of the gradient oracle (CPU only): what fixes dL/dparameter other
than the oracle's own chain rule.

* Central finite differences of the float64 loss on a tiny model, for
  entries of every parameter tensor (truncation error O(h^2) ~ 1e-10 at
  h = 1e-5, rounding ~1e-11 / h): a dropped path, a wrong sign, a missing
  1/N or a transposed operand moves a derivative by far more than 1e-6.
* torch autograd in float64 on an independently written module stack
  (a different derivation of the same derivatives), for every tensor, with
  both GPT2Config switches off and on and n_inner != 4 D.
* Invariants the pages name (llm.c notes 5.3): the LayerNorm input gradient
  is orthogonal to the constant vector and to x - mean (LN's output does not
  change under a shift or a scaling of its input row), dbeta = sum dy and
  dgamma = sum dy * xhat; the softmax-score gradient of each row sums to zero
  and is exactly zero at the causally masked positions, so no later key or
  value receives gradient from an earlier query.
"""
import math

import numpy as np
import pytest

import oracle as O
from synth import Dims, draw_model, draw_tokens


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# ------------------------------------------------------------- LayerNorm
def test_layer_norm_backward_invariants():
    r = _rng(1)
    x = r.standard_normal((7, 24)) * 3 + 1.5
    g = 1 + 0.3 * r.standard_normal(24)
    dy = r.standard_normal((7, 24))
    for eps in (1e-5, 0.3):
        dx, dg, db = O.layer_norm_backward(dy, x, g, eps)
        xc = x - x.mean(-1, keepdims=True)
        var = (xc ** 2).mean(-1, keepdims=True)
        xhat = xc / np.sqrt(var + eps)
        # a shift of the row leaves LN unchanged: dx is orthogonal to 1
        assert np.max(np.abs(dx.sum(-1))) < 1e-12 * np.abs(dx).sum()
        # a scaling by (1 + a) moves LN by a * gamma * xhat * eps / (var + eps)
        # (to first order): sum dx (x - mu) = eps / (var + eps) sum dy gamma xhat
        lhs = (dx * xc).sum(-1)
        rhs = (eps / (var + eps))[:, 0] * (dy * g * xhat).sum(-1)
        np.testing.assert_allclose(lhs, rhs, rtol=1e-9, atol=1e-13)
        np.testing.assert_allclose(db, dy.sum(0), rtol=0, atol=1e-14)
        np.testing.assert_allclose(dg, (dy * xhat).sum(0), rtol=1e-13, atol=1e-14)
    # eps -> 0: scale invariance, dx orthogonal to x - mu as well
    dx0, _, _ = O.layer_norm_backward(dy, x, g, 0.0)
    xc = x - x.mean(-1, keepdims=True)
    assert np.max(np.abs((dx0 * xc).sum(-1))) < 1e-12 * np.abs(dx0 * xc).sum()


def test_layer_norm_backward_against_finite_differences():
    r = _rng(2)
    x = r.standard_normal((3, 16))
    g, b = 1 + 0.2 * r.standard_normal(16), 0.1 * r.standard_normal(16)
    w = r.standard_normal((3, 16))  # L = sum(w * LN(x))
    dx, dg, db = O.layer_norm_backward(w, x, g, 1e-5)
    h = 1e-6
    for (i, j) in [(0, 0), (1, 5), (2, 15)]:
        xp, xm = x.copy(), x.copy()
        xp[i, j] += h
        xm[i, j] -= h
        fd = ((w * O.layer_norm(xp, g, b, 1e-5)).sum() - (w * O.layer_norm(xm, g, b, 1e-5)).sum()) / (2 * h)
        assert abs(fd - dx[i, j]) < 1e-7 * max(1.0, abs(fd))


# -------------------------------------------------------------------- GELU
@pytest.mark.parametrize("exact", [False, True])
def test_gelu_backward_values(exact):
    torch = pytest.importorskip("torch")
    u = np.linspace(-6, 6, 241)
    got = (O.gelu_exact_backward if exact else O.gelu_new_backward)(np.ones_like(u), u)
    t = torch.tensor(u, dtype=torch.float64, requires_grad=True)
    torch.nn.functional.gelu(t, approximate="none" if exact else "tanh").sum().backward()
    np.testing.assert_allclose(got, t.grad.numpy(), rtol=1e-12, atol=1e-14)
    # GELU'(0) = 1/2 for both forms; the derivative tends to 1 and 0 at the ends
    at0 = (O.gelu_exact_backward if exact else O.gelu_new_backward)(np.ones(1), np.zeros(1))[0]
    assert abs(at0 - 0.5) < 1e-15
    assert abs(got[-1] - 1) < 1e-6 and abs(got[0]) < 1e-6


# --------------------------------------------------------------- attention
def test_attention_backward_masked_and_causal():
    """dS is zero at every masked position and each row of dS sums to zero;
    a gradient at query i reaches only the keys and values of positions <= i."""
    r = _rng(3)
    B, T, H, hd = 1, 9, 2, 4
    qkv = r.standard_normal((B, T, 3 * H * hd))
    i = 4
    dout = np.zeros((B, T, H * hd))
    dout[:, i] = r.standard_normal(H * hd)
    dqkv = O.causal_attention_backward(dout, qkv, H)
    D = H * hd
    dk, dv = dqkv[..., D:2 * D], dqkv[..., 2 * D:]
    assert np.all(dk[:, i + 1:] == 0) and np.all(dv[:, i + 1:] == 0)
    assert np.abs(dk[:, :i + 1]).sum() > 0 and np.abs(dv[:, :i + 1]).sum() > 0
    # rows of dS: recompute the pieces the oracle uses
    q, k, v = O.split_qkv_heads(qkv, H)
    p = O.causal_probs(q, k)
    dout_full = r.standard_normal((B, T, D))
    do = dout_full.reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    dp = do @ np.swapaxes(v, -1, -2)
    ds = p * (dp - (dp * p).sum(-1, keepdims=True))
    assert np.max(np.abs(ds.sum(-1))) < 1e-12
    assert np.all(np.triu(ds[0, 0], 1) == 0)


@pytest.mark.parametrize("extra", [1.0, 1.0 / 3.0])
def test_attention_backward_against_torch(extra):
    torch = pytest.importorskip("torch")
    r = _rng(4)
    B, T, H, hd = 2, 11, 3, 8
    D = H * hd
    qkv = r.standard_normal((B, T, 3 * D))
    dout = r.standard_normal((B, T, D))
    got = O.causal_attention_backward(dout, qkv, H, extra)
    t = torch.tensor(qkv, dtype=torch.float64, requires_grad=True)
    q, k, v = t.split(D, dim=-1)
    sh = lambda a: a.view(B, T, H, hd).transpose(1, 2)  # noqa: E731
    o = torch.nn.functional.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True,
                                                         scale=extra / math.sqrt(hd))
    (o.transpose(1, 2).reshape(B, T, D) * torch.tensor(dout)).sum().backward()
    np.testing.assert_allclose(got, t.grad.numpy(), rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------- whole model
TINY = Dims(n_layer=2, d_model=8, n_head=2, d_ff=32, vocab=13, n_pos=7)


def _tiny(seed, **kw):
    import dataclasses
    dims = dataclasses.replace(TINY, **kw)
    params, d = draw_model(dims, "f32", seed)
    # float64 copies: the finite differences perturb entries in place
    params = {k: (v if k == "blocks" else np.asarray(v, np.float64)) for k, v in params.items()}
    params["blocks"] = [{k: np.asarray(v, np.float64) for k, v in b.items()} for b in params["blocks"]]
    # larger weights than the N(0, 0.02) recipe, so that every path of the
    # tiny model carries gradient well above the finite-difference error
    r = _rng(seed + 100)
    for blk in params["blocks"]:
        for key in ("w_qkv", "w_o", "w_fc", "w_proj"):
            blk[key] = blk[key] * 25.0
        for key in ("ln1_g", "ln2_g"):
            blk[key] = blk[key] + 0.3 * r.standard_normal(blk[key].shape)
    params["wte"] = params["wte"] * 25.0
    params["wpe"] = params["wpe"] * 25.0
    tokens = draw_tokens(d, 2, 6, dims.vocab)
    labels = tokens  # the usual next-token loss: the labels are the ids (shifted inside)
    return dims, params, tokens, labels


def _entries(params, r, per_tensor=2):
    """(path, index) of a few entries of every tensor."""
    out = []
    for key in ("wte", "wpe", "lnf_g", "lnf_b"):
        a = params[key]
        for _ in range(per_tensor):
            out.append(((key,), tuple(int(r.integers(0, n)) for n in a.shape)))
    for l, blk in enumerate(params["blocks"]):
        for key, a in blk.items():
            for _ in range(per_tensor):
                out.append((("blocks", l, key), tuple(int(r.integers(0, n)) for n in a.shape)))
    return out


def _get(tree, path):
    for p in path:
        tree = tree[p]
    return tree


@pytest.mark.parametrize("switches", [(False, False), (True, True)])
def test_loss_gradients_against_finite_differences(switches):
    inv, ge = switches
    dims, params, tokens, labels = _tiny(11, scale_attn_by_inverse_layer_idx=inv, gelu_exact=ge,
                                         d_ff=24 if ge else 32)
    loss, grads = O.loss_and_grads(tokens, labels, params, dims)
    _, _, ref_loss = O.forward_loss(tokens, labels, params, dims)
    assert abs(loss - ref_loss) < 1e-12
    r = _rng(12)
    h = 1e-5
    worst = 0.0
    for path, idx in _entries(params, r):
        a = _get(params, path)
        old = a[idx]
        a[idx] = old + h
        lp = O.forward_loss(tokens, labels, params, dims)[2]
        a[idx] = old - h
        lm = O.forward_loss(tokens, labels, params, dims)[2]
        a[idx] = old
        fd = (lp - lm) / (2 * h)
        an = _get(grads, path)[idx]
        err = abs(fd - an) / max(1e-3, abs(fd))
        worst = max(worst, err)
        assert err < 1e-5, (path, idx, fd, an)
    assert worst < 1e-5


@pytest.mark.parametrize("switches", [(False, False), (True, True)])
def test_loss_gradients_against_torch_autograd(switches):
    torch = pytest.importorskip("torch")
    Fn = torch.nn.functional
    inv, ge = switches
    dims, params, tokens, labels = _tiny(21, scale_attn_by_inverse_layer_idx=inv, gelu_exact=ge,
                                         d_ff=24 if ge else 32)
    loss, grads = O.loss_and_grads(tokens, labels, params, dims)

    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)  # noqa: E731
    P = {k: t(v) for k, v in params.items() if k != "blocks"}
    P["blocks"] = [{k: t(v) for k, v in b.items()} for b in params["blocks"]]
    B, T = tokens.shape
    D, H = dims.d_model, dims.n_head
    hd = D // H
    tok = torch.tensor(tokens, dtype=torch.long)
    x = P["wte"][tok] + P["wpe"][:T]
    for l, b in enumerate(P["blocks"]):
        a = Fn.layer_norm(x, (D,), b["ln1_g"], b["ln1_b"], dims.eps)
        q, k, v = torch.addmm(b["b_qkv"], a.reshape(-1, D), b["w_qkv"]).view(B, T, 3 * D).split(D, dim=-1)
        sh = lambda z: z.view(B, T, H, hd).transpose(1, 2)  # noqa: E731
        sc = 1.0 / math.sqrt(hd) / ((l + 1) if inv else 1)
        o = Fn.scaled_dot_product_attention(sh(q), sh(k), sh(v), is_causal=True, scale=sc)
        o = o.transpose(1, 2).reshape(B * T, D)
        x = x + torch.addmm(b["b_o"], o, b["w_o"]).view(B, T, D)
        a2 = Fn.layer_norm(x, (D,), b["ln2_g"], b["ln2_b"], dims.eps).reshape(-1, D)
        g = Fn.gelu(torch.addmm(b["b_fc"], a2, b["w_fc"]), approximate="none" if ge else "tanh")
        x = x + torch.addmm(b["b_proj"], g, b["w_proj"]).view(B, T, D)
    z = Fn.layer_norm(x, (D,), P["lnf_g"], P["lnf_b"], dims.eps) @ P["wte"].T
    lt = Fn.cross_entropy(z[:, :-1].reshape(-1, dims.vocab), torch.tensor(labels[:, 1:], dtype=torch.long).reshape(-1))
    lt.backward()
    assert abs(float(lt.detach()) - loss) < 1e-12
    for key in ("wte", "wpe", "lnf_g", "lnf_b"):
        np.testing.assert_allclose(grads[key], P[key].grad.numpy(), rtol=1e-9, atol=1e-12, err_msg=key)
    for l, b in enumerate(P["blocks"]):
        for key, tt in b.items():
            np.testing.assert_allclose(grads["blocks"][l][key], tt.grad.numpy(), rtol=1e-9, atol=1e-12,
                                       err_msg=f"block {l} {key}")


def test_tied_head_and_embedding_both_reach_wte():
    """wte collects the lm_head gradient for every row (all logits) and the
    embedding gradient only for the ids used: rows of ids absent from the
    batch get the head's part alone."""
    dims, params, tokens, labels = _tiny(31)
    loss, grads = O.loss_and_grads(tokens, labels, params, dims)
    absent = sorted(set(range(dims.vocab)) - set(tokens.reshape(-1).tolist()))
    assert absent, "the tiny batch uses every id"
    # head-only gradient of wte: dz^T LN_f(x_L)
    xL = O.forward_hidden(tokens, params, dims)
    xf = O.layer_norm(xL, params["lnf_g"], params["lnf_b"], dims.eps)
    z = xf @ params["wte"].T
    n = tokens.shape[0] * (tokens.shape[1] - 1)
    dz = np.exp(z - O.logsumexp(z)[..., None]) / n
    dz[:, -1] = 0
    for b in range(tokens.shape[0]):
        for t in range(tokens.shape[1] - 1):
            dz[b, t, labels[b, t + 1]] -= 1.0 / n
    head = dz.reshape(-1, dims.vocab).T @ xf.reshape(-1, dims.d_model)
    np.testing.assert_allclose(grads["wte"][absent], head[absent], rtol=1e-12, atol=1e-15)
    used = sorted(set(tokens.reshape(-1).tolist()))
    assert np.abs(grads["wte"][used] - head[used]).max() > 1e-6
    # positions beyond T get no gradient
    assert np.all(grads["wpe"][tokens.shape[1]:] == 0)
