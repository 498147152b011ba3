"""Oracle: a plain, slow float64 CPU statement of the GPT-2 Pre-LN forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library.

Every function follows the equations of the pages directly, in float64, with
numpy's matmul as the only library primitive.  Inputs are widened to float64
on entry; there is no intermediate rounding.  Sources (page title, section):

* "Hidden State 如何流过 GPT-2 Block" -- block dataflow (section "GPT-2 Block":
  A = Attention(LN_attn(X)), H = X + A, M = MLP(LN_ffn(H)), X' = H + M),
  LayerNorm formula (section "Pre-Norm"), stacking (section "12 个 Block").
* "逐行拆GPT-2源码" -- GPT2Config (eps = 1e-5, 4*D inner size), Conv1D
  weights stored [in, out] and applied as bias + x @ W (GPT2Attention
  section), the Q|K|V split and the 64-wide heads (``_split_heads``), the
  ``_attn`` scores / sqrt(head_dim) with future positions masked and a
  softmax, ``_merge_heads``, gelu_new (GPT2MLP section), learned absolute
  positions starting at past_length, the KV cache concatenated along the
  sequence axis, and the tied lm_head (GPT2LMHeadModel section).
* llm.c notes (page 5), sections 2.2-2.3 (scale 1/sqrt(d_k), mask before the
  softmax, max subtraction), 3.2 (LayerNorm: mean, variance, eps added to the
  variance inside the square root) and 4.2 (tanh form of GELU).

Readings where the pages are silent or disagree (listed again in the design
notes): the LayerNorm variance is the biased one (divide by D); masked scores
are excluded exactly (every masked constant the pages give yields the same
float64 result because the diagonal is always visible); the attention scale
has no layer-index factor; dropout is the identity (inference); the lm_head
is tied to wte; argmax ties go to the lowest index.

Parity pins for each function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import math

import numpy as np

F64 = np.float64


def _f64(a):
    return np.asarray(a, dtype=F64)


# ---------------------------------------------------------------- LayerNorm
def layer_norm(x, gamma, beta, eps):
    """LN(x) = gamma * (x - mu) / sqrt(var + eps) + beta over the last axis.

    "Hidden State 如何流过 GPT-2 Block", section "Pre-Norm" (the LN formula);
    llm.c notes section 3.2 (two passes: mean, then variance; eps inside the
    square root).  The variance divides by D (population variance).
    """
    x = _f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return _f64(gamma) * (x - mu) / np.sqrt(var + eps) + _f64(beta)


# ------------------------------------------------------------------ gelu_new
def gelu_new(x):
    """0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).

    "逐行拆GPT-2源码", GPT2MLP section (NewGELUActivation); llm.c notes 4.2.
    """
    x = _f64(x)
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


def gelu_exact(x):
    """x * Phi(x) = 0.5 x (1 + erf(x / sqrt(2))), Phi the standard normal CDF.

    llm.c notes 4.2 (GELU is x times the normal CDF; the tanh form above is
    its usual approximation).  The MLP uses it when the model's
    ``gelu_exact`` switch is on.
    """
    x = _f64(x)
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def _erf(x):
    return np.vectorize(math.erf, otypes=[F64])(x)


# ------------------------------------------------------------------- Conv1D
def conv1d(x, w, b):
    """Hugging Face Conv1D: bias + x @ W with W stored [in, out].

    "逐行拆GPT-2源码", GPT2Attention section (c_attn / c_proj).
    """
    return _f64(x) @ _f64(w) + _f64(b)


# ---------------------------------------------------------------- attention
def split_qkv_heads(qkv, n_head):
    """[B, T, 3D] -> Q, K, V each [B, H, T, hd].

    ``split(split_size, dim=2)`` gives Q = columns [0, D), K = [D, 2D),
    V = [2D, 3D); ``_split_heads`` views each as [B, T, H, hd] and permutes
    to [B, H, T, hd] ("逐行拆GPT-2源码", GPT2Attention section).
    """
    qkv = _f64(qkv)
    B, T, D3 = qkv.shape
    D = D3 // 3
    hd = D // n_head
    q, k, v = qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:]

    def heads(t):
        return t.reshape(B, T, n_head, hd).transpose(0, 2, 1, 3)

    return heads(q), heads(k), heads(v)


def merge_heads(o):
    """[B, H, T, hd] -> [B, T, H*hd] (``_merge_heads``)."""
    B, H, T, hd = o.shape
    return o.transpose(0, 2, 1, 3).reshape(B, T, H * hd)


def causal_probs(q, k, extra_scale=1.0):
    """softmax over j <= i of q_i . k_j / sqrt(hd), per head.

    "逐行拆GPT-2源码", ``_attn``: scores = Q K^T / sqrt(value.size(-1)); the
    causal mask keeps j <= i before the softmax; llm.c notes 2.2-2.3 (mask
    before the softmax, subtract the row maximum).  Masked scores are set to
    -inf so that exp() of them is exactly 0.
    q: [..., Tq, hd] for query positions (Tk - Tq) .. Tk-1; k: [..., Tk, hd].
    """
    q, k = _f64(q), _f64(k)
    hd = q.shape[-1]
    Tq, Tk = q.shape[-2], k.shape[-2]
    s = (q @ np.swapaxes(k, -1, -2)) / math.sqrt(hd) * extra_scale
    qpos = np.arange(Tk - Tq, Tk)[:, None]
    kpos = np.arange(Tk)[None, :]
    s = np.where(kpos <= qpos, s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def causal_attention(qkv, n_head, extra_scale=1.0):
    """Multi-head causal self-attention on packed QKV [B, T, 3D] -> [B, T, D].

    extra_scale multiplies the scores after the 1/sqrt(hd) scale ("逐行拆GPT-2
    源码", GPT2Config section: with scale_attn_by_inverse_layer_idx each
    layer's scores are further divided by layer_idx + 1).
    """
    q, k, v = split_qkv_heads(qkv, n_head)
    p = causal_probs(q, k, extra_scale)
    return merge_heads(p @ v)


# -------------------------------------------------------------------- block
def attn_extra_scale(layer, scale_attn_by_inverse_layer_idx):
    """1 / (layer + 1) with the switch on, else 1 (layer counted from 0)."""
    return 1.0 / (layer + 1) if scale_attn_by_inverse_layer_idx else 1.0


def block_forward(x, blk, n_head, eps, layer=0, scale_attn_by_inverse_layer_idx=False, gelu_exact_mlp=False):
    """One Pre-LN block, [B, T, D] -> [B, T, D].

    "Hidden State 如何流过 GPT-2 Block", section "GPT-2 Block":
    A = Attention(LN_attn(X)); H = X + A; M = MLP(LN_ffn(H)); X' = H + M.
    Attention = c_proj(merge(softmax-attention(split(c_attn(.))))) and
    MLP = c_proj(gelu_new(c_fc(.))) ("逐行拆GPT-2源码", GPT2Block / GPT2MLP).
    The two GPT2Config switches change the attention scale of layer
    ``layer`` and the MLP activation (gelu_exact).
    """
    x = _f64(x)
    a = layer_norm(x, blk["ln1_g"], blk["ln1_b"], eps)
    qkv = conv1d(a, blk["w_qkv"], blk["b_qkv"])
    o = causal_attention(qkv, n_head, attn_extra_scale(layer, scale_attn_by_inverse_layer_idx))
    h = x + conv1d(o, blk["w_o"], blk["b_o"])
    return h + mlp_forward(layer_norm(h, blk["ln2_g"], blk["ln2_b"], eps), blk, gelu_exact_mlp)


def mlp_forward(a, blk, gelu_exact_mlp=False):
    """MLP on an already-normalised input: c_proj(act(c_fc(a))), act gelu_new
    (or the exact GELU with the switch on)."""
    act = gelu_exact if gelu_exact_mlp else gelu_new
    return conv1d(act(conv1d(a, blk["w_fc"], blk["b_fc"])), blk["w_proj"], blk["b_proj"])


def _switches(dims):
    return (getattr(dims, "scale_attn_by_inverse_layer_idx", False), getattr(dims, "gelu_exact", False))


# ------------------------------------------------------------ whole model
def embed(tokens, wte, wpe, pos0=0):
    """x0[b, t] = wte[tokens[b, t]] + wpe[pos0 + t] (learned absolute positions).

    "逐行拆GPT-2源码", GPT2Model section (wte, wpe; position_ids start at
    past_length).
    """
    tokens = np.asarray(tokens)
    T = tokens.shape[-1]
    return _f64(wte)[tokens] + _f64(wpe)[pos0:pos0 + T]


def forward_hidden(tokens, params, dims):
    """Embedding, then the stack of blocks; returns the final residual stream."""
    x = embed(tokens, params["wte"], params["wpe"])
    inv, ge = _switches(dims)
    for l, blk in enumerate(params["blocks"]):
        x = block_forward(x, blk, dims.n_head, dims.eps, l, inv, ge)
    return x


def lm_head(x, params, dims):
    """logits = LN_f(x) @ wte^T (tied, no bias).

    "逐行拆GPT-2源码", GPT2LMHeadModel section (lm_head shares wte);
    "Transformer Stack" page: final LayerNorm then the output head.
    """
    return layer_norm(x, params["lnf_g"], params["lnf_b"], dims.eps) @ _f64(params["wte"]).T


def forward_logits(tokens, params, dims):
    """[B, T] token ids -> [B, T, V] logits."""
    return lm_head(forward_hidden(tokens, params, dims), params, dims)


def argmax_lowest(logits):
    """Greedy choice over the last axis; ties go to the lowest index."""
    return np.argmax(_f64(logits), axis=-1)  # numpy returns the first maximum


# ------------------------------------------------------------------- loss
def logsumexp(z):
    """log sum_v exp(z_v) over the last axis, with the row maximum taken out
    first so that no exponential overflows (llm.c notes section 2.3, the
    max subtraction of the softmax)."""
    z = _f64(z)
    m = z.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]


def shifted_cross_entropy(logits, labels):
    """The language-model loss of GPT2LMHeadModel.

    "逐行拆GPT-2源码", GPT2LMHeadModel section: the logits of positions
    0 .. T-2 are scored against the labels of positions 1 .. T-1 (the shift
    happens inside, so the labels may be the input ids themselves), each
    position by the cross-entropy -log softmax(z)[label] = lse(z) - z[label],
    and the mean is taken over all B (T-1) positions (the default reduction
    of CrossEntropyLoss).  Labels must lie in [0, V).

    Returns (token_loss [B, T-1], lse [B, T], mean).
    """
    logits = _f64(logits)
    labels = np.asarray(labels)
    B, T, V = logits.shape
    if T < 2:
        raise ValueError("the shifted loss needs T >= 2")
    if labels.shape != (B, T) or labels.min() < 0 or labels.max() >= V:
        raise ValueError("labels must be [B, T] ids in [0, V)")
    lse = logsumexp(logits)
    nxt = labels[:, 1:]
    z_t = np.take_along_axis(logits[:, :-1, :], nxt[..., None], axis=-1)[..., 0]
    token_loss = lse[:, :-1] - z_t
    return token_loss, lse, float(token_loss.mean())


def forward_loss(tokens, labels, params, dims):
    """Forward over [B, T] tokens, then the shifted cross-entropy against
    labels (labels = tokens for the usual next-token loss)."""
    return shifted_cross_entropy(forward_logits(tokens, params, dims), labels)


# ----------------------------------------------------------------- decode
def decode_step(params, dims, cache, past_len, tokens):
    """One KV-cache decode step for every sequence of the batch.

    cache: float [L, 2, B, H, T_max, hd] (K at index 0, V at index 1); slots
    < past_len[b] hold the earlier positions of sequence b.  The new token of
    sequence b sits at position past_len[b] ("逐行拆GPT-2源码", GPT2Model:
    position_ids start at past_length).  Per layer its k, v rows are appended
    at slot past_len[b] (the ``torch.cat`` along the sequence axis of
    GPT2Attention) and its query attends over slots 0 .. past_len[b].

    Returns (next_tokens [B], logits [B, V], new_cache, past_len + 1).  The
    input cache is not modified.
    """
    cache = np.array(cache, dtype=F64, copy=True)
    past_len = np.asarray(past_len)
    tokens = np.asarray(tokens)
    B = tokens.shape[0]
    D, H = dims.d_model, dims.n_head
    hd = D // H
    x = np.stack([_f64(params["wte"])[tokens[b]] + _f64(params["wpe"])[past_len[b]] for b in range(B)])
    inv, ge = _switches(dims)
    for l, blk in enumerate(params["blocks"]):
        a = layer_norm(x, blk["ln1_g"], blk["ln1_b"], dims.eps)
        qkv = conv1d(a, blk["w_qkv"], blk["b_qkv"])
        o = np.zeros((B, D))
        for b in range(B):
            p = past_len[b]
            q = qkv[b, :D].reshape(H, 1, hd)
            cache[l, 0, b, :, p, :] = qkv[b, D:2 * D].reshape(H, hd)
            cache[l, 1, b, :, p, :] = qkv[b, 2 * D:].reshape(H, hd)
            k = cache[l, 0, b, :, :p + 1, :]
            v = cache[l, 1, b, :, :p + 1, :]
            pr = causal_probs(q, k, attn_extra_scale(l, inv))  # the query is the last position
            o[b] = (pr @ v).reshape(D)
        h = x + conv1d(o, blk["w_o"], blk["b_o"])
        x = h + mlp_forward(layer_norm(h, blk["ln2_g"], blk["ln2_b"], dims.eps), blk, ge)
    logits = lm_head(x, params, dims)
    return argmax_lowest(logits), logits, cache, past_len + 1


def prefill_cache(tokens, params, dims, T_max):
    """Run a full forward and keep each layer's K, V as a cache [L,2,B,H,T_max,hd]."""
    tokens = np.asarray(tokens)
    B, T = tokens.shape
    D, H = dims.d_model, dims.n_head
    hd = D // H
    cache = np.zeros((dims.n_layer, 2, B, H, T_max, hd))
    x = embed(tokens, params["wte"], params["wpe"])
    inv, ge = _switches(dims)
    for l, blk in enumerate(params["blocks"]):
        a = layer_norm(x, blk["ln1_g"], blk["ln1_b"], dims.eps)
        qkv = conv1d(a, blk["w_qkv"], blk["b_qkv"])
        _, k, v = split_qkv_heads(qkv, H)
        cache[l, 0, :, :, :T] = k
        cache[l, 1, :, :, :T] = v
        x = block_forward(x, blk, H, dims.eps, l, inv, ge)
    return cache
