"""The language-model loss (shifted cross-entropy) on the GPU against the oracle.

Tolerance, derived from the arithmetic: lse is 1-Lipschitz in the max norm
(|lse(z + d) - lse(z)| <= max|d|), so a position's loss lse(z) - z[label]
moves by at most 2 max_v |d_v| when its logits move by d.  The GPU's logits
differ from the oracle's by the bf16 rounding of the GEMM inputs; each
position's loss is held to 2 max_v |z_gpu - z_oracle| of that position (the
GPU logits from gpt2_forward_logits, which runs the same forward) plus the
fp32 evaluation of lse (1e-5 relative).  Separately, the fused path (log-sum-
exp partials in the lm_head's epilogue, logits never stored) must equal the
loss computed in float64 from the GPU's own fp32 logits to fp32 rounding:
both come from the same GEMM, so this pins the epilogue's bookkeeping
(labels, shift, column slices, the vocabulary edge) exactly.
"""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_util import to_np

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


class _Model:
    def __init__(self, dims, dtype, params):
        self.dims, self.dt = dims, (G.BF16 if dtype == "bf16" else G.F16 if dtype == "f16" else G.F32)
        self.dev = G.to_device(params, self.dt)
        self.mw, self.keep = G.model_weights(self.dev)
        self.cd = G.make_dims(dims.n_layer, dims.d_model, dims.n_head, dims.d_ff, dims.vocab, dims.n_pos, dims.eps,
                              self.dt)

    def loss(self, tokens, labels=None):
        B, T = tokens.shape
        tl = torch.full((B, T - 1), float("nan"), device="cuda")
        lse = torch.full((B, T), float("nan"), device="cuda")
        mean = torch.full((1,), float("nan"), device="cuda")
        wsb = G.gpt2_loss_workspace_bytes(self.cd, B, T)
        ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
        tok = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).cuda()
        lab = None if labels is None else torch.from_numpy(np.ascontiguousarray(labels, np.int32)).cuda()
        G.gpt2_forward_loss(self.cd, self.mw, tok, lab, tl, lse, mean, B, T, ws, wsb)
        torch.cuda.synchronize()
        return to_np(tl), to_np(lse), float(mean.item())

    def logits(self, tokens):
        B, T = tokens.shape
        ld = (self.dims.vocab + 7) // 8 * 8
        out = torch.empty(B, T, ld, device="cuda", dtype=torch.float32)
        wsb = G.gpt2_workspace_bytes(self.cd, B, T)
        ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
        tok = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).cuda()
        G.gpt2_forward_logits(self.cd, self.mw, tok, out, ld, G.F32, B, T, ws, wsb)
        torch.cuda.synchronize()
        return to_np(out[..., :self.dims.vocab])


def _check(m, tokens, labels, ref_logits, rows=None):
    """GPU loss vs (a) float64 from the GPU's own logits (tight) and (b) the
    oracle (2 max|dz| per position)."""
    tl, lse, mean = m.loss(tokens, labels)
    lab = tokens if labels is None else labels
    z = m.logits(tokens).astype(np.float64)
    own_tl, own_lse, own_mean = O.shifted_cross_entropy(z, lab)
    np.testing.assert_allclose(lse, own_lse, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(tl, own_tl, rtol=1e-5, atol=2e-5)
    assert abs(mean - own_mean) <= 1e-5 * abs(own_mean) + 1e-5
    rows = range(tokens.shape[0]) if rows is None else rows
    for i, b in enumerate(rows):
        r_tl, r_lse, _ = O.shifted_cross_entropy(ref_logits[i:i + 1], lab[b:b + 1])
        dz = np.abs(z[b] - ref_logits[i]).max(-1)  # [T]
        bound = 2 * dz[:-1] + 1e-5 * np.abs(r_tl[0]) + 1e-5
        assert np.all(np.abs(tl[b] - r_tl[0]) <= bound), np.max(np.abs(tl[b] - r_tl[0]) - bound)
        assert np.all(np.abs(lse[b] - r_lse[0]) <= dz + 1e-5 * np.abs(r_lse[0]) + 1e-5)
    return tl, lse, mean


@pytest.mark.parametrize("B,T", [(2, 150), (1, 200), (3, 7), (1, 64)],
                         ids=["pair-kernel", "one-sm-kernel", "few-rows", "few-rows-64"])
def test_loss_bf16_paths(B, T):
    """M = B T rows picks the lm_head kernel: 300 -> CTA pair (fused), 200 ->
    single-CTA tiles (fused), 21 and 64 -> the few-row GEMM with stored
    logits."""
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2)
    params, d = synth.draw_model(dims, "bf16", 41 + T)
    tokens = synth.draw_tokens(d, B, T, dims.vocab)
    ref = O.forward_logits(tokens, params, dims)
    _check(_Model(dims, "bf16", params), tokens, None, ref)


def test_loss_separate_labels_and_ragged_vocab():
    """Labels other than the inputs, including the last vocabulary column
    and column 0; a vocabulary that ends inside a column slice."""
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=1, vocab=5003)
    params, d = synth.draw_model(dims, "bf16", 8)
    tokens = synth.draw_tokens(d, 2, 160, dims.vocab)
    labels = synth.draw_tokens(d, 2, 160, dims.vocab)
    labels[0, 1::7] = dims.vocab - 1
    labels[1, 2::5] = 0
    ref = O.forward_logits(tokens, params, dims)
    _check(_Model(dims, "bf16", params), tokens, labels, ref)


def test_loss_f16_path():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2, vocab=8000)
    params, d = synth.draw_model(dims, "bf16", 12)
    params = synth.convert_params(params, "f16")
    tokens = synth.draw_tokens(d, 2, 140, dims.vocab)
    ref = O.forward_logits(tokens, params, dims)
    _check(_Model(dims, "f16", params), tokens, None, ref)


def test_loss_fp32_path():
    """The fp32 model: the loss matches the oracle to the fp32 gate (1e-4 of
    the loss), with no bf16 rounding anywhere."""
    dims = synth.Dims(n_layer=2, d_model=128, n_head=2, d_ff=512, vocab=1000, n_pos=64)
    params, d = synth.draw_model(dims, "f32", 7)
    tokens = synth.draw_tokens(d, 2, 50, dims.vocab)
    tl, lse, mean = _Model(dims, "f32", params).loss(tokens)
    r_tl, r_lse, r_mean = O.forward_loss(tokens, tokens, params, dims)
    np.testing.assert_allclose(tl, r_tl, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(lse, r_lse, rtol=1e-5)
    assert abs(mean - r_mean) <= 1e-4 * abs(r_mean)


def test_loss_is_deterministic():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=1)
    params, d = synth.draw_model(dims, "bf16", 3)
    tokens = synth.draw_tokens(d, 4, 128, dims.vocab)
    m = _Model(dims, "bf16", params)
    a, b = m.loss(tokens), m.loss(tokens)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]


def test_loss_label_out_of_range_is_reported():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=1, vocab=3000)
    params, d = synth.draw_model(dims, "bf16", 2)
    tokens = synth.draw_tokens(d, 2, 100, dims.vocab)
    labels = tokens.copy()
    labels[1, 40] = dims.vocab  # scores position 39 of sequence 1
    labels[0, 0] = -5           # position 0's label is never used
    tl, _, mean = _Model(dims, "bf16", params).loss(tokens, labels)
    st, site = G.gpt2_last_error()
    assert st == 6 and site == 17
    assert np.isnan(tl[1, 39]) and np.isnan(mean)
    assert np.isfinite(np.delete(tl.reshape(-1), 99 + 39)).all()


def test_loss_argument_errors():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=1, vocab=300)
    params, d = synth.draw_model(dims, "bf16", 2)
    m = _Model(dims, "bf16", params)
    tok = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    out = torch.empty(4, device="cuda")
    ws = torch.empty(1 << 20, device="cuda", dtype=torch.uint8)
    with pytest.raises(G.GPT2Error):  # T = 1: no position has a next label
        G.gpt2_forward_loss(m.cd, m.mw, tok, None, None, None, out, 1, 1, ws, 1 << 20)
    tok = torch.zeros(1, 8, dtype=torch.int32, device="cuda")
    with pytest.raises(G.GPT2Error):  # no output
        G.gpt2_forward_loss(m.cd, m.mw, tok, None, None, None, None, 1, 8, ws, 1 << 20)
    with pytest.raises(G.GPT2Error):  # workspace too small
        G.gpt2_forward_loss(m.cd, m.mw, tok, None, None, None, out, 1, 8, ws, 16)


def test_loss_gpt2_small_full_size():
    """GPT-2 small, B=8, T=1024 (the forward benchmark's batch): the fused
    path over all 8192 positions; the oracle checks sequences 0 and 7."""
    inp = synth.workload_inputs("gpt2_small_fwd_b8_t1024")
    dims, params, tokens = inp["dims"], inp["params"], inp["tokens"]
    ref = np.concatenate([O.forward_logits(tokens[b:b + 1], params, dims) for b in (0, 7)], axis=0)
    tl, _, mean = _check(_Model(dims, "bf16", params), tokens, None, ref, rows=(0, 7))
    assert abs(mean - tl.mean(dtype=np.float64)) <= 1e-6 * abs(mean)
