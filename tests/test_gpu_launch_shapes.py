"""Element-wise parity at the launch shapes of the GPT-2 small forward
(B = 8, T = 1024: M = 8192 rows), the configuration the benchmark times.

At these sizes the GEMMs run persistent: the CTA-pair kernel walks several
256 x 256 tiles per pair through its double-buffered tensor-memory
accumulators (c_attn: 288 tiles, c_fc: 384, the lm_head: 6304 over 76 pairs),
and the single-CTA kernel several 128 x BN tiles per CTA (the two D-wide
projections); the attention kernel walks 768 (sequence, head, query-tile)
items over its persistent CTAs.  Smaller parity tests reach one tile per CTA
at most, so these compare every output (the lm_head: two rows of every
256-row tile, all 50257 columns) with the oracle at the shapes that run in
the forward, with the epilogue each launch has there:

  c_attn       y = a W_qkv + b        [8192, 768] x [768, 2304] -> bf16
  attn c_proj  h = x + o W_o + b      [8192, 768] x [768, 768]  -> fp32
  c_fc         g = gelu_new(a W + b)  [8192, 768] x [768, 3072] -> bf16
  mlp c_proj   x = h + g W_p + b      [8192, 3072] x [3072, 768] -> fp32
  lm_head      z = a wte^T            [8192, 768] x [50257, 768]^T -> fp32 / bf16
  attention    softmax(q k^T / 8, j <= i) v, B = 8, T = 1024, 12 heads

The bounds are those of the smaller kernel tests (derived there): output
rounding (2^-8 relative for bf16, 2^-20 for fp32), 2^-14 sum |a w| of fp32
accumulation, 2^-11 |z| for the hardware tanh of gelu_new, and 2^-8 sum_j
p_j |v_j| for the bf16 probabilities of the attention.
"""
import numpy as np
import pytest

import oracle as O
from gpu_util import assert_close_elementwise, bf16, f32, rng, to_np, to_t

torch = pytest.importorskip("torch")
import gpt_pre_ln_gb300 as G  # noqa: E402

pytestmark = pytest.mark.gpu

M = 8192  # B * T of the forward


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gpt_pre_ln_gb300 import build
    build.build()
    G.lib()
    yield
    st, site = G.gpt2_last_error()
    assert st == 0, f"device error {st} at site {site}"


LAYER_GEMMS = [
    # name, N, K, epilogue
    ("c_attn", 2304, 768, G.EPI_BIAS),
    ("attn_c_proj", 768, 768, G.EPI_BIAS_RESIDUAL),
    ("c_fc", 3072, 768, G.EPI_BIAS_GELU),
    ("mlp_c_proj", 768, 3072, G.EPI_BIAS_RESIDUAL),
]


@pytest.mark.parametrize("name,N,K,epi", LAYER_GEMMS, ids=[c[0] for c in LAYER_GEMMS])
def test_layer_gemm_at_forward_shape(name, N, K, epi):
    r = rng(N * 3 + K)
    x = bf16(r.standard_normal((M, K)))
    w = bf16(0.02 * r.standard_normal((K, N)))
    bias = bf16(0.5 * r.standard_normal(N))
    res = f32(r.standard_normal((M, N)))
    y_t = "f32" if epi == G.EPI_BIAS_RESIDUAL else "bf16"
    y = torch.full((M, N), float("nan"), device="cuda", dtype=torch.float32 if y_t == "f32" else torch.bfloat16)
    G.gpt2_linear(to_t(x, "bf16"), to_t(w, "bf16"), to_t(bias, "bf16"), to_t(res, "f32"), y, M, N, K, N,
                  G.W_IN_OUT, epi, G.BF16, G.F32 if y_t == "f32" else G.BF16)
    torch.cuda.synchronize()
    got = to_np(y)
    x64, w64 = x.astype(np.float64), w.astype(np.float64)
    pre = x64 @ w64 + bias
    absz = np.abs(x64) @ np.abs(w64)
    ref = pre
    if epi == G.EPI_BIAS_GELU:
        ref = O.gelu_new(pre)
    if epi == G.EPI_BIAS_RESIDUAL:
        ref = pre + res
    rtol = 2.0 ** -8 if y_t == "bf16" else 2.0 ** -20
    bound = rtol * np.abs(ref) + 2.0 ** -14 * absz * 1.2 + 1e-30
    if epi == G.EPI_BIAS_GELU:
        bound = bound + 2.0 ** -11 * np.abs(pre)
    assert_close_elementwise(got, ref, bound, name)


@pytest.mark.parametrize("y_t", ["f32", "bf16"])
def test_lm_head_at_forward_shape(y_t):
    V, D = 50257, 768
    r = rng(50257 + (y_t == "bf16"))
    a = bf16(r.standard_normal((M, D)))
    wte = bf16(0.02 * r.standard_normal((V, D)))
    ld = (V + 7) // 8 * 8
    y = torch.empty(M, ld, device="cuda", dtype=torch.float32 if y_t == "f32" else torch.bfloat16)
    G.gpt2_linear(to_t(a, "bf16"), to_t(wte, "bf16"), None, None, y, M, V, D, ld, G.W_OUT_IN, G.EPI_NONE, G.BF16,
                  G.F32 if y_t == "f32" else G.BF16)
    torch.cuda.synchronize()
    # one row in each 128-row half of every 256-row tile of the CTA pair
    rows = np.array([t * 128 + int(r.integers(0, 128)) for t in range(M // 128)])
    got = to_np(y[torch.from_numpy(rows).cuda(), :V])
    w64 = wte.astype(np.float64)
    ref = a[rows].astype(np.float64) @ w64.T
    absz = np.abs(a[rows].astype(np.float64)) @ np.abs(w64).T
    rtol = 2.0 ** -8 if y_t == "bf16" else 2.0 ** -20
    assert_close_elementwise(got, ref, rtol * np.abs(ref) + 2.0 ** -14 * absz * 1.2 + 1e-30, f"lm_head {y_t}")


def test_attention_at_forward_shape():
    B, T, H = 8, 1024, 12
    D = 64 * H
    r = rng(8 * 1024)
    qkv = bf16(r.standard_normal((B, T, 3 * D)) * 1.5)
    out = torch.full((B, T, D), float("nan"), device="cuda", dtype=torch.bfloat16)
    G.gpt2_attention_causal(to_t(qkv, "bf16"), out, B, T, H, 64, G.BF16)
    torch.cuda.synchronize()
    got = to_np(out)
    for b in range(B):  # the oracle one sequence at a time (memory)
        ref = O.causal_attention(qkv[b:b + 1], H)
        q, k, v = O.split_qkv_heads(qkv[b:b + 1], H)
        pav = O.merge_heads(O.causal_probs(q, k) @ np.abs(v))
        assert_close_elementwise(got[b:b + 1], ref, 2.0 ** -8 * np.abs(ref) + 2.0 ** -8 * pav + 1e-6,
                                 f"attention sequence {b}")
