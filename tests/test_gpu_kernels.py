"""Per-kernel parity on the GPU: each C-ABI entry point against the oracle.

Inputs are seeded and already exact in the path dtype, so both sides see
the same numbers; the oracle then computes in float64 without intermediate
rounding.  Each bound below is derived from the arithmetic of the kernel:

* bf16 outputs are rounded to nearest: |error| <= 2^-9 |y|; the bounds use
  2^-8 |y| (a factor two of slack).
* fp32 accumulation of K products (exact in fp32 for bf16 inputs) adds at
  most a few units of 2^-24 per term in practice; the bounds use
  2^-14 * sum_k |a_k w_k|, far below what a wrong term would change.
* gelu_new on a bf16 output uses the hardware tanh (absolute error below
  2^-11): an extra 2^-11 |z| on the pre-activation z.
* attention rounds the probabilities to bf16 before P.V: an extra
  2^-8 * sum_j p_j |v_j|.
"""
import numpy as np
import pytest

import oracle as O
from gpu_util import assert_close_elementwise, bf16, f32, max_rel_err, rng, to_np, to_t

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


# ------------------------------------------------------------------ LayerNorm
@pytest.mark.parametrize("D", [64, 768, 1024, 1600])
@pytest.mark.parametrize("y_t", ["bf16", "f32"])
def test_layernorm(D, y_t):
    r = rng(100 + D)
    rows = 333
    x = f32(r.standard_normal((rows, D)) * 3 + 0.5)
    g = (bf16 if y_t == "bf16" else f32)(1 + 0.2 * r.standard_normal(D))
    b = (bf16 if y_t == "bf16" else f32)(0.2 * r.standard_normal(D))
    xt = to_t(x, "f32")
    y = torch.empty(rows, D, device="cuda", dtype=torch.bfloat16 if y_t == "bf16" else torch.float32)
    yt_code = G.BF16 if y_t == "bf16" else G.F32
    G.gpt2_layernorm(xt, to_t(g, y_t), to_t(b, y_t), y, rows, D, 1e-5, G.F32, yt_code)
    torch.cuda.synchronize()
    ref = O.layer_norm(x, g, b, 1e-5)
    got = to_np(y)
    if y_t == "bf16":
        assert_close_elementwise(got, ref, 2.0 ** -8 * np.abs(ref) + 1e-5, "layernorm bf16")
    else:
        assert_close_elementwise(got, ref, 1e-5 * np.abs(ref) + 1e-5, "layernorm f32")


def test_layernorm_bf16_input_and_empty():
    r = rng(5)
    x = bf16(r.standard_normal((70, 768)))
    g, b = bf16(1 + 0.1 * r.standard_normal(768)), bf16(0.1 * r.standard_normal(768))
    y = torch.empty(70, 768, device="cuda", dtype=torch.bfloat16)
    G.gpt2_layernorm(to_t(x, "bf16"), to_t(g, "bf16"), to_t(b, "bf16"), y, 70, 768, 1e-5, G.BF16, G.BF16)
    G.gpt2_layernorm(None, None, None, None, 0, 768, 1e-5, G.F32, G.BF16)  # empty: no-op
    torch.cuda.synchronize()
    ref = O.layer_norm(x, g, b, 1e-5)
    assert_close_elementwise(to_np(y), ref, 2.0 ** -8 * np.abs(ref) + 1e-5, "layernorm bf16 in")


# --------------------------------------------------------------------- linear
LINEAR_CASES = [
    # (M, N, K, layout)
    (333, 768, 768, G.W_IN_OUT),      # attention c_proj shape, ragged M
    (200, 2304, 768, G.W_IN_OUT),     # c_attn
    (129, 3072, 768, G.W_IN_OUT),     # c_fc, M one past a tile
    (257, 768, 3072, G.W_IN_OUT),     # mlp c_proj (K = 4D)
    (1, 256, 64, G.W_IN_OUT),         # single row, single k-block
    (300, 1000, 768, G.W_OUT_IN),     # lm_head style, ragged N
    (520, 1000, 768, G.W_IN_OUT),     # ragged N in the last 192-wide pair tile, W read N-major
    (300, 3072, 768, G.W_IN_OUT),     # c_fc shape over two 256-row pair units (the second ragged)
    (130, 50257, 768, G.W_OUT_IN),    # full vocabulary
    # few rows (one token per sequence of a decode step): the swapped-operand
    # kernel with K split over a thread-block cluster
    (16, 8, 64, G.W_IN_OUT),          # one partial tile, one k-block
    (7, 2304, 768, G.W_IN_OUT),       # c_attn, 18 tiles
    (33, 200, 192, G.W_IN_OUT),       # ragged N in the second tile, 3 k-blocks
    (64, 768, 768, G.W_IN_OUT),       # attention c_proj at a decode batch of 64
    (64, 768, 3072, G.W_IN_OUT),      # mlp c_proj
    (64, 3072, 768, G.W_IN_OUT),      # c_fc
    (100, 1000, 768, G.W_OUT_IN),     # wte layout, ragged N
    (128, 768, 768, G.W_IN_OUT),      # the largest row count of this kernel
    (64, 50257, 768, G.W_OUT_IN),     # lm_head of a decode step: persistent over 393 tiles
    (64, 4800, 1600, G.W_IN_OUT),     # XL c_attn: N not a multiple of 256
]


def _linear_ref(x, w, bias, res, epi, layout):
    wm = w if layout == G.W_IN_OUT else w.T
    z = x.astype(np.float64) @ wm.astype(np.float64)
    absz = np.abs(x.astype(np.float64)) @ np.abs(wm.astype(np.float64))
    if epi != G.EPI_NONE:
        z = z + bias
    pre = z
    if epi == G.EPI_BIAS_GELU:
        z = O.gelu_new(z)
    if epi == G.EPI_BIAS_RESIDUAL:
        z = z + res
    return z, absz, pre


@pytest.mark.parametrize("case", LINEAR_CASES, ids=lambda c: f"M{c[0]}N{c[1]}K{c[2]}L{c[3]}")
@pytest.mark.parametrize("epi", [G.EPI_NONE, G.EPI_BIAS, G.EPI_BIAS_GELU, G.EPI_BIAS_RESIDUAL])
def test_linear_bf16(case, epi):
    M, N, K, layout = case
    if N == 50257 and epi != G.EPI_NONE:
        pytest.skip("the lm_head has no bias")
    r = rng(M * 7 + N + K + epi)
    x = bf16(r.standard_normal((M, K)))
    w = bf16(0.02 * r.standard_normal((K, N) if layout == G.W_IN_OUT else (N, K)))
    bias = bf16(0.5 * r.standard_normal(N))
    res = f32(r.standard_normal((M, N)))
    y_t = "f32" if epi == G.EPI_BIAS_RESIDUAL else "bf16"
    ld = (N + 15) // 8 * 8 if layout == G.W_OUT_IN else N  # padded row stride (at least 8 spare columns)
    y = torch.full((M, ld), float("nan"), device="cuda", dtype=torch.float32 if y_t == "f32" else torch.bfloat16)
    rt = to_t(res, "f32")
    G.gpt2_linear(to_t(x, "bf16"), to_t(w, "bf16"), to_t(bias, "bf16"), rt, y, M, N, K, ld, layout, epi, G.BF16,
                  G.F32 if y_t == "f32" else G.BF16)
    torch.cuda.synchronize()
    got = to_np(y)
    esz = 4 if y_t == "f32" else 2
    n16 = (N * esz + 15) // 16 * 16 // esz  # the row padding up to 16 bytes is written with zeros
    assert np.all(got[:, N:n16] == 0), "padding up to the 16-byte boundary"
    assert np.all(np.isnan(got[:, n16:])), "wrote past the 16-byte boundary after N"
    got = got[:, :N]
    ref, absz, pre = _linear_ref(x, w, bias, res, epi, layout)
    rtol = 2.0 ** -8 if y_t == "bf16" else 2.0 ** -20
    bound = rtol * np.abs(ref) + 2.0 ** -14 * absz * 1.2 + 1e-30
    if epi == G.EPI_BIAS_GELU:
        bound = bound + 2.0 ** -11 * np.abs(pre)
    assert_close_elementwise(got, ref, bound, f"linear epi={epi}")


@pytest.mark.parametrize("M,N,K", [(64, 768, 3072), (5, 2304, 768), (64, 50257, 768)])
def test_linear_few_rows_is_deterministic(M, N, K):
    """The split-K partial sums are added in a fixed order: two calls give
    the same bits."""
    r = rng(M + N)
    layout = G.W_OUT_IN if N == 50257 else G.W_IN_OUT
    x = to_t(bf16(r.standard_normal((M, K))), "bf16")
    w = to_t(bf16(0.02 * r.standard_normal((K, N) if layout == G.W_IN_OUT else (N, K))), "bf16")
    ld = (N + 3) // 4 * 4
    ys = []
    for _ in range(2):
        y = torch.empty(M, ld, device="cuda", dtype=torch.float32)
        G.gpt2_linear(x, w, None, None, y, M, N, K, ld, layout, G.EPI_NONE, G.BF16, G.F32)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(ys[0][:, :N], ys[1][:, :N])


@pytest.mark.parametrize("epi", [G.EPI_BIAS, G.EPI_BIAS_GELU, G.EPI_BIAS_RESIDUAL])
def test_linear_f32(epi):
    M, N, K = 77, 300, 192
    r = rng(epi)
    x = f32(r.standard_normal((M, K)))
    w = f32(0.05 * r.standard_normal((K, N)))
    bias = f32(r.standard_normal(N))
    res = f32(r.standard_normal((M, N)))
    y = torch.empty(M, N, device="cuda")
    G.gpt2_linear(to_t(x, "f32"), to_t(w, "f32"), to_t(bias, "f32"), to_t(res, "f32"), y, M, N, K, N, G.W_IN_OUT,
                  epi, G.F32, G.F32)
    torch.cuda.synchronize()
    ref, absz, _ = _linear_ref(x, w, bias, res, epi, G.W_IN_OUT)
    assert_close_elementwise(to_np(y), ref, 2.0 ** -20 * np.abs(ref) + 2.0 ** -18 * absz, "linear f32")


def test_linear_in_place_residual():
    """y may be the residual buffer itself (x' = h + ... written over h)."""
    M, N, K = 140, 768, 768
    r = rng(9)
    x = bf16(r.standard_normal((M, K)))
    w = bf16(0.02 * r.standard_normal((K, N)))
    bias = bf16(r.standard_normal(N))
    res = f32(r.standard_normal((M, N)))
    rt = to_t(res, "f32")
    G.gpt2_linear(to_t(x, "bf16"), to_t(w, "bf16"), to_t(bias, "bf16"), rt, rt, M, N, K, N, G.W_IN_OUT,
                  G.EPI_BIAS_RESIDUAL, G.BF16, G.F32)
    torch.cuda.synchronize()
    ref, absz, _ = _linear_ref(x, w, bias, res, G.EPI_BIAS_RESIDUAL, G.W_IN_OUT)
    assert_close_elementwise(to_np(rt), ref, 2.0 ** -20 * np.abs(ref) + 2.0 ** -14 * absz, "in place")


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("T", [1, 17, 64, 65, 200, 1024])
def test_attention_bf16(T):
    B, H = 2, 12
    D = 64 * H
    r = rng(T)
    qkv = bf16(r.standard_normal((B, T, 3 * D)) * 1.5)
    out = torch.full((B, T, D), float("nan"), device="cuda", dtype=torch.bfloat16)
    G.gpt2_attention_causal(to_t(qkv, "bf16"), out, B, T, H, 64, G.BF16)
    torch.cuda.synchronize()
    ref = O.causal_attention(qkv, H)
    q, k, v = O.split_qkv_heads(qkv, H)
    pav = O.merge_heads(O.causal_probs(q, k) @ np.abs(v))
    assert_close_elementwise(to_np(out), ref, 2.0 ** -8 * np.abs(ref) + 2.0 ** -8 * pav + 1e-6, f"attention T={T}")


@pytest.mark.parametrize("T", [1, 33, 64, 130])
def test_attention_f32(T):
    B, H = 2, 3
    D = 64 * H
    r = rng(50 + T)
    qkv = f32(r.standard_normal((B, T, 3 * D)))
    out = torch.empty(B, T, D, device="cuda")
    G.gpt2_attention_causal(to_t(qkv, "f32"), out, B, T, H, 64, G.F32)
    torch.cuda.synchronize()
    ref = O.causal_attention(qkv, H)
    assert max_rel_err(to_np(out), ref) < 1e-5


def test_attention_causality_on_gpu():
    """Changing keys/values after position i leaves outputs 0..i bit-identical."""
    B, T, H = 1, 200, 12
    D = 64 * H
    r = rng(77)
    qkv = bf16(r.standard_normal((B, T, 3 * D)))
    out1 = torch.empty(B, T, D, device="cuda", dtype=torch.bfloat16)
    out2 = torch.empty_like(out1)
    G.gpt2_attention_causal(to_t(qkv, "bf16"), out1, B, T, H, 64, G.BF16)
    qkv2 = qkv.copy()
    i = 130
    qkv2[:, i + 1:] = bf16(r.standard_normal((B, T - i - 1, 3 * D)))
    G.gpt2_attention_causal(to_t(qkv2, "bf16"), out2, B, T, H, 64, G.BF16)
    torch.cuda.synchronize()
    assert torch.equal(out1[:, :i + 1], out2[:, :i + 1])
    assert not torch.equal(out1[:, i + 1:], out2[:, i + 1:])


@pytest.mark.parametrize("growth", [0.05, 0.5])
def test_attention_rising_scores(growth):
    """Keys whose scale grows along the sequence, so that a row's running
    maximum keeps rising by more than the kernel's rescale threshold (8 in
    log2 units) from chunk to chunk and tile to tile: every rescale path (the
    accumulated output, the sums, and the probabilities already written for
    the tile's first chunk) runs; the output and the row log-sum-exps stay
    within the bounds of the plain case."""
    B, T, H = 2, 400, 3
    D = 64 * H
    r = rng(1300 + int(growth * 100))
    qkv = r.standard_normal((B, T, 3 * D))
    qkv[:, :, D:2 * D] *= (1.0 + growth * np.arange(T))[None, :, None] / 4.0
    qkv = bf16(qkv)
    out = torch.full((B, T, D), float("nan"), device="cuda", dtype=torch.bfloat16)
    lse = torch.full((B, H, T), float("nan"), device="cuda")
    G.gpt2_attention_causal_lse(to_t(qkv, "bf16"), out, lse, B, T, H, 64, 0.125, G.BF16)
    torch.cuda.synchronize()
    ref = O.causal_attention(qkv, H)
    q, k, v = O.split_qkv_heads(qkv, H)
    pav = O.merge_heads(O.causal_probs(q, k) @ np.abs(v))
    assert_close_elementwise(to_np(out), ref, 2.0 ** -8 * np.abs(ref) + 2.0 ** -8 * pav + 1e-6, f"growth {growth}")
    s_ = (q @ np.swapaxes(k, -1, -2)) / 8.0
    s_ = np.where(np.tril(np.ones((T, T), bool)), s_, -np.inf)
    ref_lse = O.logsumexp(s_) / np.log(2.0)
    # each score is an fp32 sum of 64 exact products: |error| <= 64 u sum |q_d k_d| / 8
    # (u = 2^-24), in log2 units; the log-sum-exp moves by at most the largest
    # of its scores' errors (plus fp32 rounding of its own, 1e-4)
    sabs = (np.abs(q) @ np.swapaxes(np.abs(k), -1, -2)) / 8.0
    sabs = np.where(np.tril(np.ones((T, T), bool)), sabs, 0.0)
    bound = 1e-4 + 2.0 * 64 * 2.0 ** -24 * sabs.max(-1) / np.log(2.0)
    assert np.all(np.abs(to_np(lse) - ref_lse) <= bound)
    # the scores of the last rows span far more than the threshold
    assert (s_[:, :, -1, :].max(-1) - s_[:, :, -1, :64].max(-1)).max() / np.log(2.0) > 8.0


# ------------------------------------------------------------------------ MLP
@pytest.mark.parametrize("with_res", [True, False])
def test_mlp_bf16(with_res):
    M, D, F = 150, 768, 3072
    r = rng(31)
    x = bf16(r.standard_normal((M, D)))
    w_fc, b_fc = bf16(0.02 * r.standard_normal((D, F))), bf16(0.01 * r.standard_normal(F))
    w_p, b_p = bf16(0.004 * r.standard_normal((F, D))), bf16(0.01 * r.standard_normal(D))
    res = f32(r.standard_normal((M, D)))
    out = torch.empty(M, D, device="cuda")
    wsb = G.gpt2_mlp_workspace_bytes(M, F, G.BF16)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_mlp(to_t(x, "bf16"), to_t(w_fc, "bf16"), to_t(b_fc, "bf16"), to_t(w_p, "bf16"), to_t(b_p, "bf16"),
               to_t(res, "f32") if with_res else None, out, M, D, F, ws, wsb, G.BF16)
    torch.cuda.synchronize()
    blk = {"w_fc": w_fc, "b_fc": b_fc, "w_proj": w_p, "b_proj": b_p}
    ref = O.mlp_forward(x, blk) + (res if with_res else 0)
    delta = O.mlp_forward(x, blk)
    # the hidden activation is rounded to bf16 (2^-9 relative) before c_proj
    g_abs = np.abs(O.gelu_new(x @ w_fc.astype(np.float64) + b_fc))
    bound = 2.0 ** -8 * (g_abs @ np.abs(w_p.astype(np.float64))) + 2.0 ** -20 * np.abs(ref) + 1e-6
    assert_close_elementwise(to_np(out), ref, bound, "mlp")
    assert np.abs(delta).max() > 1e-3  # the MLP contributes


def test_workspace_too_small_is_reported():
    with pytest.raises(G.GPT2Error) as e:
        dummy = torch.empty(64, device="cuda")
        ws = torch.empty(256, device="cuda", dtype=torch.uint8)
        G.gpt2_mlp(dummy, dummy, dummy, dummy, dummy, None, dummy, 4, 64, 256, ws, 256, G.BF16)
    assert e.value.status == 3
