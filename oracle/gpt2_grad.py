"""Oracle: the gradients of the GPT-2 language-model loss, in float64 on the CPU.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module: only ``tests/`` use it.  It shares no code with the CUDA
library; the forward pieces it differentiates are those of ``gpt2_ref``.

Backpropagation is written out step by step, in reverse order of the
forward, with numpy's matmul as the only library primitive:

* llm.c notes, section 5.2: every intermediate of the forward is kept for
  the backward pass (here: recomputed from the saved block inputs).
* llm.c notes, section 5.3: the LayerNorm gradient couples the mean, the
  variance and the normalised value, and gamma and beta have gradients of
  their own; the softmax gradient follows the max-subtracted forward; the
  gradient at causally masked positions is zero and is set to zero
  explicitly.
* "逐行拆GPT-2源码", GPT2LMHeadModel section: the loss is the mean
  cross-entropy of positions 0 .. T-2 against the labels of positions
  1 .. T-1, and the lm_head shares wte with the embedding, so wte collects
  the gradient of both uses.

Parity pins are in ``tests/test_oracle_grad_pins.py`` (central finite
differences, torch autograd in float64, and the invariants of the LayerNorm
and softmax gradients).
"""
from __future__ import annotations

import math

import numpy as np

from .gpt2_ref import (attn_extra_scale, block_forward, causal_probs, conv1d, embed, gelu_exact, gelu_new,
                       layer_norm, logsumexp, merge_heads, split_qkv_heads)

F64 = np.float64


def _f64(a):
    return np.asarray(a, dtype=F64)


# ---------------------------------------------------------------- LayerNorm
def layer_norm_backward(dy, x, gamma, eps):
    """Gradients of y = gamma * (x - mu) / sqrt(var + eps) + beta.

    llm.c notes 5.3: dx collects three paths -- through the normalised value
    directly, through the variance and through the mean; dgamma = sum of
    dy * xhat and dbeta = sum of dy over every row.  Returns
    (dx, dgamma, dbeta).
    """
    x, dy, gamma = _f64(x), _f64(dy), _f64(gamma)
    D = x.shape[-1]
    mu = x.mean(axis=-1, keepdims=True)
    xc = x - mu
    var = (xc ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = xc * rstd
    dxhat = dy * gamma
    # var = mean(xc^2), rstd = (var + eps)^(-1/2)
    dvar = (dxhat * xc).sum(axis=-1, keepdims=True) * (-0.5) * rstd ** 3
    # mu enters xhat directly and through var (whose mu-gradient
    # mean(-2 xc) vanishes identically; kept as the chain rule gives it)
    dmu = (-dxhat * rstd).sum(axis=-1, keepdims=True) + dvar * (-2.0 * xc).mean(axis=-1, keepdims=True)
    dx = dxhat * rstd + dvar * 2.0 * xc / D + dmu / D
    rows = dy.reshape(-1, D)
    dgamma = (rows * xhat.reshape(-1, D)).sum(axis=0)
    dbeta = rows.sum(axis=0)
    return dx, dgamma, dbeta


# --------------------------------------------------------------------- GELU
def gelu_new_backward(dy, u):
    """d/du of 0.5 u (1 + tanh(k (u + 0.044715 u^3))), k = sqrt(2/pi)."""
    u = _f64(u)
    k = math.sqrt(2.0 / math.pi)
    t = np.tanh(k * (u + 0.044715 * u ** 3))
    return _f64(dy) * (0.5 * (1.0 + t) + 0.5 * u * (1.0 - t * t) * k * (1.0 + 3.0 * 0.044715 * u * u))


def gelu_exact_backward(dy, u):
    """d/du of u Phi(u) = Phi(u) + u phi(u), phi the standard normal density."""
    u = _f64(u)
    Phi = 0.5 * (1.0 + np.vectorize(math.erf, otypes=[F64])(u / math.sqrt(2.0)))
    phi = np.exp(-0.5 * u * u) / math.sqrt(2.0 * math.pi)
    return _f64(dy) * (Phi + u * phi)


# ------------------------------------------------------------------- Conv1D
def conv1d_backward(dy, x, w):
    """y = b + x @ W (W [in, out]): dx = dy W^T, dW = x^T dy and db = sum of
    dy, both summed over every row."""
    dy, x, w = _f64(dy), _f64(x), _f64(w)
    dx = dy @ w.T
    dw = x.reshape(-1, x.shape[-1]).T @ dy.reshape(-1, dy.shape[-1])
    db = dy.reshape(-1, dy.shape[-1]).sum(axis=0)
    return dx, dw, db


# ---------------------------------------------------------------- attention
def causal_attention_backward(dout, qkv, n_head, extra_scale=1.0):
    """Gradient of the packed QKV [B, T, 3D] given that of the merged output.

    With s = q k^T * c (c = extra_scale / sqrt(hd)), p = softmax over the
    visible keys and o = p v:  dv = p^T do,  dp = do v^T,
    ds = p * (dp - sum_j dp_j p_j)  (the softmax Jacobian; the row maximum
    subtracted in the forward cancels out of it), ds = 0 at the masked
    positions (llm.c notes 5.3: set explicitly), dq = c ds k, dk = c ds^T q.
    """
    q, k, v = split_qkv_heads(qkv, n_head)
    B, H, T, hd = q.shape
    c = extra_scale / math.sqrt(hd)
    p = causal_probs(q, k, extra_scale)
    do = _f64(dout).reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    dv = np.swapaxes(p, -1, -2) @ do
    dp = do @ np.swapaxes(v, -1, -2)
    ds = p * (dp - (dp * p).sum(axis=-1, keepdims=True))
    visible = np.arange(T)[None, :] <= np.arange(T)[:, None]
    ds = np.where(visible, ds, 0.0)
    dq = c * (ds @ k)
    dk = c * (np.swapaxes(ds, -1, -2) @ q)
    return np.concatenate([merge_heads(dq), merge_heads(dk), merge_heads(dv)], axis=-1)


# -------------------------------------------------------------------- block
def block_backward(dx_out, x, blk, n_head, eps, layer=0, scale_attn_by_inverse_layer_idx=False,
                   gelu_exact_mlp=False):
    """Backward through one Pre-LN block given dL/dX' and the block input X.

    Forward (recomputed): a = LN_1(x); qkv = c_attn(a); o = attention(qkv);
    h = x + c_proj(o); a2 = LN_2(h); u = c_fc(a2); g = act(u);
    x' = h + c_proj2(g).  Returns (dL/dX, {tensor name: gradient}).
    """
    x = _f64(x)
    extra = attn_extra_scale(layer, scale_attn_by_inverse_layer_idx)
    a = layer_norm(x, blk["ln1_g"], blk["ln1_b"], eps)
    qkv = conv1d(a, blk["w_qkv"], blk["b_qkv"])
    q, k, v = split_qkv_heads(qkv, n_head)
    o = merge_heads(causal_probs(q, k, extra) @ v)
    h = x + conv1d(o, blk["w_o"], blk["b_o"])
    a2 = layer_norm(h, blk["ln2_g"], blk["ln2_b"], eps)
    u = conv1d(a2, blk["w_fc"], blk["b_fc"])
    g = gelu_exact(u) if gelu_exact_mlp else gelu_new(u)

    grads = {}
    dx_out = _f64(dx_out)
    # x' = h + c_proj2(g)
    dg, grads["w_proj"], grads["b_proj"] = conv1d_backward(dx_out, g, blk["w_proj"])
    du = gelu_exact_backward(dg, u) if gelu_exact_mlp else gelu_new_backward(dg, u)
    da2, grads["w_fc"], grads["b_fc"] = conv1d_backward(du, a2, blk["w_fc"])
    dh_ln, grads["ln2_g"], grads["ln2_b"] = layer_norm_backward(da2, h, blk["ln2_g"], eps)
    dh = dx_out + dh_ln
    # h = x + c_proj(o)
    do, grads["w_o"], grads["b_o"] = conv1d_backward(dh, o, blk["w_o"])
    dqkv = causal_attention_backward(do, qkv, n_head, extra)
    da, grads["w_qkv"], grads["b_qkv"] = conv1d_backward(dqkv, a, blk["w_qkv"])
    dx_ln, grads["ln1_g"], grads["ln1_b"] = layer_norm_backward(da, x, blk["ln1_g"], eps)
    return dh + dx_ln, grads


# --------------------------------------------------------------- whole model
def loss_and_grads(tokens, labels, params, dims):
    """Mean shifted cross-entropy of the whole model and its gradient with
    respect to every parameter (same nesting as ``params``).

    dL/dz at position t < T-1 is (softmax(z) - onehot(labels[t+1])) / N,
    N = B (T-1), and zero at the last position of each sequence.  The tied
    lm_head logits = LN_f(x_L) wte^T give wte the gradient dz^T LN_f(x_L);
    the embedding x0 = wte[tokens] + wpe[t] adds dx0 to the rows of the
    tokens used and to the positions.
    """
    tokens = np.asarray(tokens)
    labels = np.asarray(labels)
    B, T = tokens.shape
    V = dims.vocab
    inv = getattr(dims, "scale_attn_by_inverse_layer_idx", False)
    ge = getattr(dims, "gelu_exact", False)
    wte = _f64(params["wte"])

    # forward, keeping each block's input
    xs = [embed(tokens, wte, params["wpe"])]
    for l, blk in enumerate(params["blocks"]):
        xs.append(block_forward(xs[-1], blk, dims.n_head, dims.eps, l, inv, ge))
    xf = layer_norm(xs[-1], params["lnf_g"], params["lnf_b"], dims.eps)
    z = xf @ wte.T
    lse = logsumexp(z)
    nxt = labels[:, 1:]
    z_t = np.take_along_axis(z[:, :-1, :], nxt[..., None], axis=-1)[..., 0]
    loss = float((lse[:, :-1] - z_t).mean())

    # backward
    n = B * (T - 1)
    dz = np.exp(z - lse[..., None]) / n
    dz[:, -1, :] = 0.0
    bi, ti = np.meshgrid(np.arange(B), np.arange(T - 1), indexing="ij")
    dz[bi, ti, nxt] -= 1.0 / n
    grads = {"blocks": [None] * len(params["blocks"])}
    dxf = dz @ wte
    dwte = dz.reshape(-1, V).T @ xf.reshape(-1, xf.shape[-1])
    dx, grads["lnf_g"], grads["lnf_b"] = layer_norm_backward(dxf, xs[-1], params["lnf_g"], dims.eps)
    for l in range(len(params["blocks"]) - 1, -1, -1):
        dx, grads["blocks"][l] = block_backward(dx, xs[l], params["blocks"][l], dims.n_head, dims.eps, l, inv, ge)
    # embedding
    np.add.at(dwte, tokens.reshape(-1), dx.reshape(-1, dx.shape[-1]))
    dwpe = np.zeros_like(_f64(params["wpe"]))
    dwpe[:T] = dx.sum(axis=0)
    grads["wte"] = dwte
    grads["wpe"] = dwpe
    return loss, grads

