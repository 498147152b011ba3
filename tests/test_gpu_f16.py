"""The F16 path (fp16 operands and activations, fp32 accumulation, residual
and statistics) against the oracle.

fp16 keeps 11 significant bits where bf16 keeps 8, so every rounding of the
path is 8x finer: outputs rounded to fp16 are within 2^-11 |y| (the bounds
use 2^-10), and attention probabilities within 2^-11 relative before P.V.
The model weights are the bf16 draws of the GPT-2 workloads converted to
fp16 (exact for magnitudes from 2^-17 up); the oracle uses the same values.
At the full GPT-2 small workload the F16 path is held to the acceptance
targets: logits rel L2 <= 1e-2 and top-1 agreement >= 99.5%.
"""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_util import assert_close_elementwise, f16, f32, rel_l2, rng, to_np, to_t, top1_check

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


@pytest.mark.parametrize("case", [(333, 768, 768, G.W_IN_OUT), (200, 2304, 768, G.W_IN_OUT),
                                  (257, 768, 3072, G.W_IN_OUT), (130, 50257, 768, G.W_OUT_IN),
                                  (300, 3072, 768, G.W_IN_OUT)],
                         ids=lambda c: f"M{c[0]}N{c[1]}K{c[2]}L{c[3]}")
@pytest.mark.parametrize("epi", [G.EPI_NONE, G.EPI_BIAS, G.EPI_BIAS_GELU, G.EPI_BIAS_RESIDUAL])
def test_linear_f16(case, epi):
    M, N, K, layout = case
    if N == 50257 and epi != G.EPI_NONE:
        pytest.skip("the lm_head has no bias")
    r = rng(M + N + K + 10 * epi)
    x = f16(r.standard_normal((M, K)))
    w = f16(0.02 * r.standard_normal((K, N) if layout == G.W_IN_OUT else (N, K)))
    bias = f16(0.5 * r.standard_normal(N))
    res = f32(r.standard_normal((M, N)))
    y_t = "f32" if epi in (G.EPI_BIAS_RESIDUAL, G.EPI_NONE) else "f16"
    ld = (N + 15) // 8 * 8
    y = torch.full((M, ld), float("nan"), device="cuda", dtype=torch.float32 if y_t == "f32" else torch.float16)
    G.gpt2_linear(to_t(x, "f16"), to_t(w, "f16"), to_t(bias, "f16"), to_t(res, "f32"), y, M, N, K, ld, layout, epi,
                  G.F16, G.F32 if y_t == "f32" else G.F16)
    torch.cuda.synchronize()
    got = to_np(y)[:, :N]
    wm = w.astype(np.float64) if layout == G.W_IN_OUT else w.T.astype(np.float64)
    z = x.astype(np.float64) @ wm
    absz = np.abs(x.astype(np.float64)) @ np.abs(wm)
    if epi != G.EPI_NONE:
        z = z + bias
    pre = z
    if epi == G.EPI_BIAS_GELU:
        z = O.gelu_new(z)
    if epi == G.EPI_BIAS_RESIDUAL:
        z = z + res
    rtol = 2.0 ** -10 if y_t == "f16" else 2.0 ** -20
    bound = rtol * np.abs(z) + 2.0 ** -14 * absz * 1.2 + 1e-30
    if epi == G.EPI_BIAS_GELU:
        bound = bound + 2.0 ** -11 * np.abs(pre)
    assert_close_elementwise(got, z, bound, f"linear f16 epi={epi}")


@pytest.mark.parametrize("T", [1, 65, 200, 1024])
def test_attention_f16(T):
    B, H = 2, 12
    D = 64 * H
    r = rng(700 + T)
    qkv = f16(r.standard_normal((B, T, 3 * D)) * 1.5)
    out = torch.full((B, T, D), float("nan"), device="cuda", dtype=torch.float16)
    G.gpt2_attention_causal(to_t(qkv, "f16"), out, B, T, H, 64, G.F16)
    torch.cuda.synchronize()
    ref = O.causal_attention(qkv, H)
    q, k, v = O.split_qkv_heads(qkv, H)
    pav = O.merge_heads(O.causal_probs(q, k) @ np.abs(v))
    assert_close_elementwise(to_np(out), ref, 2.0 ** -10 * np.abs(ref) + 2.0 ** -10 * pav + 1e-6, f"attn f16 T={T}")


def test_layernorm_f16():
    r = rng(3)
    x = f32(r.standard_normal((333, 768)) * 3 + 0.5)
    g, b = f16(1 + 0.2 * r.standard_normal(768)), f16(0.2 * r.standard_normal(768))
    y = torch.empty(333, 768, device="cuda", dtype=torch.float16)
    G.gpt2_layernorm(to_t(x, "f32"), to_t(g, "f16"), to_t(b, "f16"), y, 333, 768, 1e-5, G.F32, G.F16)
    torch.cuda.synchronize()
    ref = O.layer_norm(x, g, b, 1e-5)
    assert_close_elementwise(to_np(y), ref, 2.0 ** -10 * np.abs(ref) + 1e-5, "layernorm f16")


def _forward_f16(dims, params, tokens):
    B, T = tokens.shape
    dev = G.to_device(params, G.F16)
    mw, keep = G.model_weights(dev)
    cd = G.make_dims(dims.n_layer, dims.d_model, dims.n_head, dims.d_ff, dims.vocab, dims.n_pos, dims.eps, G.F16)
    ld = (dims.vocab + 7) // 8 * 8
    logits = torch.empty(B, T, ld, device="cuda", dtype=torch.float32)
    wsb = G.gpt2_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_forward_logits(cd, mw, torch.from_numpy(tokens).cuda(), logits, ld, G.F32, B, T, ws, wsb)
    torch.cuda.synchronize()
    del keep
    return logits[..., :dims.vocab]


def _check(got, ref, min_top1):
    err = rel_l2(got, ref)
    rms = float(np.sqrt(np.mean((got - ref) ** 2)))
    agree = float(np.mean(np.argmax(got, -1) == np.argmax(ref, -1)))
    print(f"F16 logits rel L2 {err:.3e}, top-1 agreement {agree:.5f}")
    assert err <= 1e-2
    top1_check(got, ref, min_top1, tie_tol=10 * rms)


def test_forward_f16_small_stack():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2)
    params, d = synth.draw_model(dims, "bf16", 99)
    tokens = synth.draw_tokens(d, 2, 150, dims.vocab)
    params = synth.convert_params(params, "f16")
    got = to_np(_forward_f16(dims, params, tokens))
    ref = O.forward_logits(tokens, params, dims)
    _check(got, ref, 0.98)


def test_forward_f16_gpt2_small_full_size():
    """GPT-2 small, B=8, T=1024, the bench workload's weights and tokens in
    fp16: the acceptance targets (rel L2 <= 1e-2, top-1 >= 99.5%) on the two
    sampled sequences (2048 positions)."""
    inp = synth.workload_inputs("gpt2_small_fwd_b8_t1024")
    dims, tokens = inp["dims"], inp["tokens"]
    params = synth.convert_params(inp["params"], "f16")
    logits = _forward_f16(dims, params, tokens)
    got = np.concatenate([to_np(logits[b:b + 1]) for b in (0, 7)], axis=1)
    ref = np.concatenate([O.forward_logits(tokens[b:b + 1], params, dims) for b in (0, 7)], axis=1)
    _check(got, ref, 0.995)


def test_decode_f16_matches_oracle():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2, n_pos=64)
    B, T_max = 3, 48
    past = np.array([5, 40, 17], np.int32)
    params, d = synth.draw_model(dims, "bf16", 11)
    params = synth.convert_params(params, "f16")
    cache = np.zeros((dims.n_layer, 2, B, dims.n_head, T_max, 64), np.float32)
    for b in range(B):
        cache[:, :, b, :, :past[b]] = f16(d.rng.standard_normal((dims.n_layer, 2, dims.n_head, past[b], 64)))
    tokens = d.rng.integers(0, dims.vocab, size=B).astype(np.int32)
    dev = G.to_device(params, G.F16)
    mw, keep = G.model_weights(dev)
    cd = G.make_dims(dims.n_layer, dims.d_model, dims.n_head, dims.d_ff, dims.vocab, dims.n_pos, dims.eps, G.F16)
    kv = to_t(cache, "f16")
    pl = torch.from_numpy(past.copy()).cuda()
    tok = torch.from_numpy(tokens.copy()).cuda()
    nxt = torch.empty_like(tok)
    ld = 50264
    logits = torch.empty(B, ld, device="cuda")
    wsb = G.gpt2_decode_workspace_bytes(cd, B)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    ocache, opast, otok = cache.astype(np.float64), past.copy(), tokens.copy()
    for _ in range(3):
        G.gpt2_decode_step(cd, mw, kv, B, T_max, pl, tok, nxt, logits, ld, ws, wsb)
        torch.cuda.synchronize()
        _, ref, ocache, opast = O.decode_step(params, dims, ocache, opast, otok)
        got = to_np(logits[:, :dims.vocab])
        assert rel_l2(got, ref) <= 2e-3
        assert np.array_equal(pl.cpu().numpy(), opast)
        otok = nxt.cpu().numpy()
        tok.copy_(nxt)
    del keep
