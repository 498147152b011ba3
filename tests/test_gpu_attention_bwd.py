"""The tensor-core causal attention backward against the gradient oracle.

gpt2_attention_causal_lse runs the forward and keeps each row's log-sum-exp;
gpt2_attention_causal_backward recomputes p from it and returns dQ | dK | dV
in the layout of qkv.  The oracle is ``causal_attention_backward`` of the
gradient oracle in float64, on the same bf16 inputs.

Bounds, derived from the arithmetic of the kernels (per element, with the
oracle's own p, ds and operands; c the score scale):
* p and ds are rounded to bf16 before they multiply (2^-9 relative each),
  the forward output o that enters delta = do . o is bf16 (2^-9 relative),
  and the outputs are rounded to bf16 (2^-9 relative); the bounds use 2^-8
  for each (a factor two of slack);
* an error e_delta in delta moves ds_qk by p_qk e_delta, with
  |e_delta| <= 2^-8 sum_d |do_qd o_qd|.
So
  |err dV_k| <= 2^-8 (|dV_k| + sum_q p_qk |do_q|)
  |err dQ_q| <= 2^-8 |dQ_q| + c (2^-8 sum_k |ds_qk| |k_k| + e_delta_q sum_k p_qk |k_k|)
  |err dK_k| <= 2^-8 |dK_k| + c (2^-8 sum_q |ds_qk| |q_q| + sum_q e_delta_q p_qk |q_q|)
"""
import math

import numpy as np
import pytest

import oracle as O
from gpu_util import assert_close_elementwise, bf16, rel_l2, rng, to_np, to_t

torch = pytest.importorskip("torch")
import gpt_pre_ln_gb300 as G  # noqa: E402
from oracle import gpt2_grad as OG  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gpt_pre_ln_gb300 import build
    build.build()
    G.lib()
    yield
    st, site = G.gpt2_last_error()
    assert st == 0, f"device error {st} at site {site}"


def _bounds(qkv, dout, H, extra):
    """Element-wise bounds on dQ | dK | dV (see the module docstring)."""
    q, k, v = O.split_qkv_heads(qkv, H)
    B, _, T, hd = q.shape
    c = extra / math.sqrt(hd)
    p = O.causal_probs(q, k, extra)
    do = dout.astype(np.float64).reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    o = p @ v
    dp = do @ np.swapaxes(v, -1, -2)
    ds = p * (dp - (dp * p).sum(-1, keepdims=True))
    e_delta = 2.0 ** -8 * (np.abs(do) * np.abs(o)).sum(-1, keepdims=True)  # [B, H, T, 1]
    dq = c * ds @ k
    dk = c * np.swapaxes(ds, -1, -2) @ q
    dv = np.swapaxes(p, -1, -2) @ do
    bq = 2.0 ** -8 * np.abs(dq) + c * (2.0 ** -8 * np.abs(ds) @ np.abs(k) + e_delta * (p @ np.abs(k)))
    bk = 2.0 ** -8 * np.abs(dk) + c * (2.0 ** -8 * np.swapaxes(np.abs(ds), -1, -2) @ np.abs(q)
                                       + np.swapaxes(p * e_delta, -1, -2) @ np.abs(q))
    bv = 2.0 ** -8 * (np.abs(dv) + np.swapaxes(p, -1, -2) @ np.abs(do))
    return np.concatenate([O.merge_heads(bq), O.merge_heads(bk), O.merge_heads(bv)], -1) + 1e-6


def _run(B, T, H, seed, extra=1.0, dtype="bf16"):
    D = 64 * H
    r = rng(seed)
    qkv = bf16(r.standard_normal((B, T, 3 * D)) * 1.5)
    dout = bf16(r.standard_normal((B, T, D)))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    code = G.BF16 if dtype == "bf16" else G.F16
    qkv_t = to_t(qkv, dtype)
    out = torch.empty(B, T, D, device="cuda", dtype=tdt)
    lse = torch.full((B, H, T), float("nan"), device="cuda")
    c = extra / 8.0
    G.gpt2_attention_causal_lse(qkv_t, out, lse, B, T, H, 64, c, code)
    dqkv = torch.full((B, T, 3 * D), float("nan"), device="cuda", dtype=tdt)
    wsb = G.gpt2_attention_backward_workspace_bytes(B, T, H)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_attention_causal_backward(qkv_t, out, lse, to_t(dout, dtype), dqkv, B, T, H, 64, c, ws, wsb, code)
    torch.cuda.synchronize()
    return qkv, dout, to_np(dqkv), to_np(lse)


@pytest.mark.parametrize("B,T,H", [(1, 1, 1), (2, 17, 2), (1, 64, 3), (2, 65, 2), (1, 128, 2), (2, 200, 3),
                                   (1, 257, 1), (2, 1024, 12)])
def test_attention_backward_bf16(B, T, H):
    qkv, dout, got, lse = _run(B, T, H, 7000 + T + B)
    ref = OG.causal_attention_backward(dout, qkv, H)
    assert np.isfinite(got).all()
    assert_close_elementwise(got, ref, _bounds(qkv, dout, H, 1.0), f"dqkv B={B} T={T} H={H}")
    D = 64 * H
    for name, sl in (("dq", slice(0, D)), ("dk", slice(D, 2 * D)), ("dv", slice(2 * D, 3 * D))):
        if np.linalg.norm(ref[..., sl]) == 0:  # T = 1: dq and dk vanish (ds = p (dp - p dp) = 0)
            assert np.all(got[..., sl] == 0), name
        else:
            assert rel_l2(got[..., sl], ref[..., sl]) < 1e-2, name


def test_attention_lse_matches_the_oracle():
    B, T, H = 2, 130, 2
    qkv, _, _, lse = _run(B, T, H, 12)
    q, k, _ = O.split_qkv_heads(qkv, H)
    s = (q @ np.swapaxes(k, -1, -2)) / 8.0
    s = np.where(np.tril(np.ones((T, T), bool)), s, -np.inf)
    ref = O.logsumexp(s) / np.log(2.0)  # log2 of the sum of e^s
    np.testing.assert_allclose(lse, ref, rtol=0, atol=1e-4)


def test_attention_backward_layer_scale_and_f16():
    """The score scale of the layer-index switch (1 / (8 (l + 1)), here l = 3)
    and the fp16 path."""
    B, T, H = 1, 190, 2
    qkv, dout, got, _ = _run(B, T, H, 31, extra=0.25)
    ref = OG.causal_attention_backward(dout, qkv, H, 0.25)
    assert_close_elementwise(got, ref, _bounds(qkv, dout, H, 0.25), "scaled")
    qkv, dout, got, _ = _run(B, T, H, 32, dtype="f16")
    ref = OG.causal_attention_backward(dout, qkv, H)
    assert_close_elementwise(got, ref, _bounds(qkv, dout, H, 1.0), "f16")


def test_attention_backward_is_deterministic():
    B, T, H = 2, 300, 2
    a = _run(B, T, H, 5)[2]
    b = _run(B, T, H, 5)[2]
    assert np.array_equal(a, b)
