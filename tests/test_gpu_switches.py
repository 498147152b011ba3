"""GPT2Config switches on the GPU against the oracle: the attention scale of
layer l divided by l + 1 (scale_attn_by_inverse_layer_idx), the exact GELU
x Phi(x) in the MLP, and n_inner (d_ff) other than 4 D.

Bounds follow the arithmetic, as in the per-kernel tests:

* the exact GELU epilogue evaluates erff in fp32 (a few fp32 ulps), so the
  fp32-output bound is the accumulation bound of the plain bias epilogue
  (2^-14 sum_k |x_k w_k|, times |GELU'| <= 1.13) plus fp32 rounding.  The
  output must also sit much closer to the exact GELU than to gelu_new
  (relative L2; the two differ by up to 4.7e-4 near |x| = 2), so an
  epilogue that kept the tanh form fails.
* bf16 outputs add 2^-8 |y| (rounding to nearest, a factor two of slack).
* attention with another score scale: the same bound as the default scale
  (probabilities rounded to bf16 before P.V: 2^-8 sum_j p_j |v_j|).
* whole-model paths: the fp32 block gate (max relative error 1e-4) and the
  bf16 logits gate (relative L2 1e-2, flipped argmaxes only at near ties).
  The switches move these logits by far more than the gate (checked), so
  a switch that is ignored fails.
"""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_util import assert_close_elementwise, bf16, f32, max_rel_err, rel_l2, rng, to_np, to_t, top1_check

torch = pytest.importorskip("torch")
import gpt_pre_ln_gb300 as G  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gpt_pre_ln_gb300 import build
    build.build()
    G.lib()
    yield
    st, site = G.gpt2_last_error()
    assert st == 0, f"device error {st} at site {site}"


def _flags(dims):
    return ((G.SCALE_ATTN_BY_INVERSE_LAYER_IDX if dims.scale_attn_by_inverse_layer_idx else 0)
            | (G.GELU_EXACT if dims.gelu_exact else 0))


def _cdims(dims, dt):
    return G.make_dims(dims.n_layer, dims.d_model, dims.n_head, dims.d_ff, dims.vocab, dims.n_pos, dims.eps, dt,
                       flags=_flags(dims))


# --------------------------------------------------------- exact GELU epilogue
@pytest.mark.parametrize("M,N,K", [(333, 3072, 768), (129, 640, 768), (64, 3072, 768), (7, 2048, 1024)])
@pytest.mark.parametrize("y_t", ["f32", "bf16"])
def test_linear_gelu_exact_bf16(M, N, K, y_t):
    """Both 16-bit GEMM kernels (tiled for M > 128, few-row otherwise)."""
    r = rng(M + N + K)
    x = bf16(r.standard_normal((M, K)))
    w = bf16(0.02 * r.standard_normal((K, N)))
    bias = bf16(0.5 * r.standard_normal(N))
    y = torch.full((M, N), float("nan"), device="cuda", dtype=torch.float32 if y_t == "f32" else torch.bfloat16)
    G.gpt2_linear(to_t(x, "bf16"), to_t(w, "bf16"), to_t(bias, "bf16"), None, y, M, N, K, N, G.W_IN_OUT,
                  G.EPI_BIAS_GELU_EXACT, G.BF16, G.F32 if y_t == "f32" else G.BF16)
    torch.cuda.synchronize()
    z = x.astype(np.float64) @ w.astype(np.float64) + bias
    absz = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64))
    ref = O.gelu_exact(z)
    bound = 2.0 ** -14 * absz * 1.2 * 1.13 + 2.0 ** -20 * np.abs(ref) + 1e-30
    if y_t == "bf16":
        bound = bound + 2.0 ** -8 * np.abs(ref)
    got = to_np(y)
    assert_close_elementwise(got, ref, bound, f"gelu_exact epilogue y={y_t}")
    if y_t == "f32":
        # the output follows the exact GELU, not the tanh form: its distance
        # from gelu_new is the GELU gap (up to 4.7e-4), far above the
        # accumulation error (rms, not the worst-case bound above)
        assert rel_l2(got, O.gelu_new(z)) > 5 * rel_l2(got, ref)


def test_linear_gelu_exact_f32():
    M, N, K = 77, 320, 192
    r = rng(4)
    x = f32(r.standard_normal((M, K)))
    w = f32(0.1 * r.standard_normal((K, N)))
    bias = f32(r.standard_normal(N))
    y = torch.empty(M, N, device="cuda")
    G.gpt2_linear(to_t(x, "f32"), to_t(w, "f32"), to_t(bias, "f32"), None, y, M, N, K, N, G.W_IN_OUT,
                  G.EPI_BIAS_GELU_EXACT, G.F32, G.F32)
    torch.cuda.synchronize()
    z = x.astype(np.float64) @ w.astype(np.float64) + bias
    absz = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64))
    ref = O.gelu_exact(z)
    bound = 2.0 ** -20 * np.abs(ref) + 2.0 ** -18 * absz * 1.13
    got = to_np(y)
    assert_close_elementwise(got, ref, bound, "gelu_exact f32")
    assert rel_l2(got, O.gelu_new(z)) > 5 * rel_l2(got, ref)


# ------------------------------------------------------------ attention scale
@pytest.mark.parametrize("T,layer", [(64, 2), (200, 11), (1024, 5)])
def test_attention_scaled_bf16(T, layer):
    B, H = 2, 12
    D = 64 * H
    r = rng(900 + T)
    qkv = bf16(r.standard_normal((B, T, 3 * D)) * 3.0)
    out = torch.full((B, T, D), float("nan"), device="cuda", dtype=torch.bfloat16)
    extra = 1.0 / (layer + 1)
    G.gpt2_attention_causal_scaled(to_t(qkv, "bf16"), out, B, T, H, 64, 0.125 * extra, G.BF16)
    torch.cuda.synchronize()
    ref = O.causal_attention(qkv, H, extra)
    q, k, v = O.split_qkv_heads(qkv, H)
    pav = O.merge_heads(O.causal_probs(q, k, extra) @ np.abs(v))
    assert_close_elementwise(to_np(out), ref, 2.0 ** -8 * np.abs(ref) + 2.0 ** -8 * pav + 1e-6,
                             f"scaled attention T={T}")
    assert rel_l2(O.causal_attention(qkv, H), ref) > 0.05  # the scale matters on this data


def test_attention_scaled_f32_and_default_equivalence():
    B, T, H = 2, 97, 3
    D = 64 * H
    r = rng(31)
    qkv = f32(r.standard_normal((B, T, 3 * D)) * 2.0)
    out = torch.empty(B, T, D, device="cuda")
    G.gpt2_attention_causal_scaled(to_t(qkv, "f32"), out, B, T, H, 64, 0.125 / 4, G.F32)
    # the unscaled entry point is the scaled one at 1/8: identical bits
    o1 = torch.empty(B, T, D, device="cuda", dtype=torch.bfloat16)
    o2 = torch.empty_like(o1)
    qb = to_t(bf16(qkv), "bf16")
    G.gpt2_attention_causal(qb, o1, B, T, H, 64, G.BF16)
    G.gpt2_attention_causal_scaled(qb, o2, B, T, H, 64, 0.125, G.BF16)
    torch.cuda.synchronize()
    assert max_rel_err(to_np(out), O.causal_attention(qkv, H, 0.25)) < 1e-5
    assert torch.equal(o1, o2)


# ----------------------------------------------------------- blocks and model
def _switched(dims, **kw):
    return synth.replace_dims(dims, scale_attn_by_inverse_layer_idx=True, gelu_exact=True, **kw)


@pytest.mark.parametrize("layer", [0, 3])
def test_block_fp32_switches_and_n_inner(layer):
    """F32 block gate (max relative error 1e-4) with both switches on and
    d_ff = 2048, at block index `layer`."""
    dims = _switched(synth.GPT2_SMALL, n_layer=1, d_ff=2048)
    params, d = synth.draw_model(dims, "f32", 77 + layer, with_embeddings=False)
    B, T = 1, 64
    x = synth.draw_activations(d, B, T, dims.d_model)
    dev = G.to_device(params, G.F32)
    cd = _cdims(dims, G.F32)
    xt = to_t(x, "f32")
    out = torch.empty_like(xt)
    wsb = G.gpt2_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_block_forward_layer(cd, G.block_weights(dev["blocks"][0]), layer, xt, out, B, T, ws, wsb)
    torch.cuda.synchronize()
    blk = params["blocks"][0]
    ref = O.block_forward(x, blk, dims.n_head, dims.eps, layer, True, True)
    got = to_np(out)
    err = max_rel_err(got, ref)
    assert err <= 1e-4, err
    # the output is much closer to the switched block than to a block with
    # either switch off (the GELU alone moves it by about 2e-4 here)
    assert max_rel_err(got, O.block_forward(x, blk, dims.n_head, dims.eps, layer, True, False)) > 5 * err
    if layer > 0:
        assert max_rel_err(got, O.block_forward(x, blk, dims.n_head, dims.eps, layer, False, True)) > 1e-2


def _bf16_model(seed, **kw):
    dims = _switched(synth.GPT2_SMALL, **kw)
    params, d = synth.draw_model(dims, "bf16", seed)
    return dims, params, d


def test_forward_bf16_switches_and_n_inner():
    """Three GPT-2 small layers with both switches and n_inner = 2048; the
    embeddings' attention scores are scaled up (x3 on the QKV weights of
    every layer) so that the per-layer scale changes the softmax visibly."""
    dims, params, d = _bf16_model(505, n_layer=3, d_ff=2048, n_pos=128)
    for blk in params["blocks"]:
        blk["w_qkv"] = bf16(blk["w_qkv"] * 3.0)
    B, T = 2, 100
    tokens = synth.draw_tokens(d, B, T, dims.vocab)
    dev = G.to_device(params, G.BF16)
    mw, keep = G.model_weights(dev)
    cd = _cdims(dims, G.BF16)
    ld = (dims.vocab + 7) // 8 * 8
    logits = torch.empty(B, T, ld, device="cuda")
    wsb = G.gpt2_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_forward_logits(cd, mw, torch.from_numpy(tokens).cuda(), logits, ld, G.F32, B, T, ws, wsb)
    torch.cuda.synchronize()
    got = to_np(logits[..., :dims.vocab])
    ref = O.forward_logits(tokens, params, dims)
    err = rel_l2(got, ref)
    assert err <= 1e-2, err
    rms = float(np.sqrt(np.mean((got - ref) ** 2)))
    top1_check(got.reshape(-1, dims.vocab), ref.reshape(-1, dims.vocab), 0.9, tie_tol=10 * rms)
    # the layer-index scale moves these logits by ~40%; the GELU switch by
    # ~1.4e-4 only, under the bf16 gate (the fp32 block and epilogue tests
    # separate the two GELUs)
    off = O.forward_logits(tokens, params, synth.replace_dims(dims, scale_attn_by_inverse_layer_idx=False))
    assert rel_l2(off, ref) > 5 * err
    del keep


def test_prefill_decode_bf16_switches():
    """Prefill writes the cache with the switched layers, and a decode step
    over it matches the oracle's step from the same cache."""
    dims, params, d = _bf16_model(606, n_layer=3, d_ff=1536, n_pos=64)
    for blk in params["blocks"]:
        blk["w_qkv"] = bf16(blk["w_qkv"] * 3.0)
    B, T, T_max = 3, 20, 40
    tokens = synth.draw_tokens(d, B, T, dims.vocab)
    dev = G.to_device(params, G.BF16)
    mw, keep = G.model_weights(dev)
    cd = _cdims(dims, G.BF16)
    kv = torch.zeros((dims.n_layer, 2, B, dims.n_head, T_max, 64), device="cuda", dtype=torch.bfloat16)
    past = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    ld = (dims.vocab + 3) // 4 * 4
    lg = torch.empty(B, ld, device="cuda")
    wsb = G.gpt2_prefill_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_prefill(cd, mw, torch.from_numpy(tokens).cuda(), B, T, kv, T_max, past, nxt, lg, ld, ws, wsb)
    torch.cuda.synchronize()
    got = to_np(lg[:, :dims.vocab])
    ref = O.forward_logits(tokens, params, dims)[:, -1]
    assert rel_l2(got, ref) <= 1e-2
    ref_cache = O.prefill_cache(tokens, params, dims, T_max)
    cache = to_np(kv)
    for l in range(dims.n_layer):
        assert rel_l2(cache[l, :, :, :, :T], ref_cache[l, :, :, :, :T]) <= 1e-2, l
    # one greedy step from the GPU's own cache, the oracle from the same cache
    step_tok = nxt.clone()
    dwsb = G.gpt2_decode_workspace_bytes(cd, B)
    dws = torch.empty(dwsb, device="cuda", dtype=torch.uint8)
    G.gpt2_decode_step(cd, mw, kv, B, T_max, past, step_tok, nxt, lg, ld, dws, dwsb)
    torch.cuda.synchronize()
    got = to_np(lg[:, :dims.vocab])
    _, ref, _, _ = O.decode_step(params, dims, cache.copy(), np.full(B, T, np.int64), step_tok.cpu().numpy())
    err = rel_l2(got, ref)
    assert err <= 1e-2, err
    assert np.all(past.cpu().numpy() == T + 1)
    off_dims = synth.replace_dims(dims, scale_attn_by_inverse_layer_idx=False, gelu_exact=False)
    _, off, _, _ = O.decode_step(params, off_dims, cache.copy(), np.full(B, T, np.int64), step_tok.cpu().numpy())
    assert rel_l2(off, ref) > 5 * err
    del keep
