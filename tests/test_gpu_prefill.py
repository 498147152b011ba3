"""Prompt prefill (forward + KV cache) and the decode steps after it, on the
GPU against the oracle.

The cache holds K and V rounded to bf16 (rms relative error 2^-8/sqrt(3),
about 1.6e-3, for the rounding alone), computed from GEMM inputs that were
rounded to bf16 in every layer before: measured 2e-3 to 4.5e-3 relative L2
per layer on these workloads.  The gate is the logits' 1e-2: K and V
swapped, a head or a position transposed, or another layer's cache all
give errors of order 1.  Slots past the prompt must be untouched bit for
bit.  The prefill's
last-position logits must also equal those of gpt2_forward_logits on the
same tokens to fp32 accumulation-order rounding: the two run the same
forward kernels, and only the lm_head (few-row kernel against the tiled
one) sums K in a different order.
"""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_util import rel_l2, to_np, top1_check

torch = pytest.importorskip("torch")
import gpt_pre_ln_gb300 as G  # noqa: E402

pytestmark = pytest.mark.gpu

SENTINEL = 3.0  # exact in bf16; what the cache holds before the prefill


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gpt_pre_ln_gb300 import build
    build.build()
    G.lib()
    yield
    st, site = G.gpt2_last_error()
    assert st == 0, f"device error {st} at site {site}"


class _Gen:
    def __init__(self, dims, params, B, T_max):
        self.dims, self.B, self.T_max = dims, B, T_max
        self.dev = G.to_device(params, G.BF16)
        self.mw, self.keep = G.model_weights(self.dev)
        self.cd = G.make_dims(dims.n_layer, dims.d_model, dims.n_head, dims.d_ff, dims.vocab, dims.n_pos, dims.eps,
                              G.BF16)
        self.kv = torch.full((dims.n_layer, 2, B, dims.n_head, T_max, 64), SENTINEL, device="cuda",
                             dtype=torch.bfloat16)
        self.past = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        self.next = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        self.ld = (dims.vocab + 3) // 4 * 4
        self.logits = torch.full((B, self.ld), float("nan"), device="cuda")

    def prefill(self, tokens):
        B, T = tokens.shape
        wsb = G.gpt2_prefill_workspace_bytes(self.cd, B, T)
        ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
        tok = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).cuda()
        G.gpt2_prefill(self.cd, self.mw, tok, B, T, self.kv, self.T_max, self.past, self.next, self.logits, self.ld,
                       ws, wsb)
        torch.cuda.synchronize()
        return to_np(self.logits[:, :self.dims.vocab])

    def decode(self):
        wsb = G.gpt2_decode_workspace_bytes(self.cd, self.B)
        ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
        tok = self.next.clone()
        G.gpt2_decode_step(self.cd, self.mw, self.kv, self.B, self.T_max, self.past, tok, self.next, self.logits,
                           self.ld, ws, wsb)
        torch.cuda.synchronize()
        return tok.cpu().numpy(), to_np(self.logits[:, :self.dims.vocab])

    def forward_last_logits(self, tokens):
        B, T = tokens.shape
        ld = (self.dims.vocab + 7) // 8 * 8
        out = torch.empty(B, T, ld, device="cuda")
        wsb = G.gpt2_workspace_bytes(self.cd, B, T)
        ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
        tok = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).cuda()
        G.gpt2_forward_logits(self.cd, self.mw, tok, out, ld, G.F32, B, T, ws, wsb)
        torch.cuda.synchronize()
        return to_np(out[:, -1, :self.dims.vocab])


def _check_prefill(g, tokens, params, dims, seqs=None):
    B, T = tokens.shape
    got = g.prefill(tokens)
    assert np.all(g.past.cpu().numpy() == T)
    # the same forward through gpt2_forward_logits: equal to fp32 rounding
    own = g.forward_last_logits(tokens)
    assert rel_l2(got, own) <= 1e-5
    nxt = g.next.cpu().numpy()
    gap = own.max(-1) - own[np.arange(B), nxt]
    assert np.all(gap <= 1e-4 * np.abs(own).max()), "argmax of the prefill's logits"
    kv = g.kv.float().cpu().numpy()
    assert np.all(kv[:, :, :, :, T:] == SENTINEL), "slots past the prompt were written"
    for b in (range(B) if seqs is None else seqs):
        ref_cache = O.prefill_cache(tokens[b:b + 1], params, dims, g.T_max)
        for l in range(dims.n_layer):
            err = rel_l2(kv[l, :, b:b + 1, :, :T], ref_cache[l, :, :, :, :T])
            assert err <= 1e-2, (b, l, err)
        ref = O.forward_logits(tokens[b:b + 1], params, dims)[:, -1]
        assert rel_l2(got[b:b + 1], ref) <= 1e-2
        top1_check(got[b:b + 1], ref, 0.0, tie_tol=10 * float(np.sqrt(np.mean((got[b] - ref) ** 2))))
    return got


def test_prefill_then_decode_matches_oracle():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2, n_pos=64)
    params, d = synth.draw_model(dims, "bf16", 21)
    B, T, T_max = 3, 20, 48
    tokens = synth.draw_tokens(d, B, T, dims.vocab)
    g = _Gen(dims, params, B, T_max)
    _check_prefill(g, tokens, params, dims)
    # greedy continuation, the oracle following the GPU's tokens: (a) the
    # whole chain from the oracle's own cache of the prompt; (b) each step
    # from the GPU's cache as it stands, so that a wrong cache and a wrong
    # step show up apart.  Both at the bf16 logits gate (1e-2; measured
    # 3-4e-3 here, the ordinary error of the 2-layer bf16 path), and the
    # chosen token must be the oracle's or a near tie.
    cache = O.prefill_cache(tokens, params, dims, T_max)
    past = np.full(B, T, np.int32)
    for _ in range(3):
        gpu_cache = g.kv.float().cpu().numpy()
        tok, got = g.decode()
        _, ref, cache, past = O.decode_step(params, dims, cache, past, tok)
        assert rel_l2(got, ref) <= 1e-2
        assert np.array_equal(g.past.cpu().numpy(), past)
        _, ref_step, _, _ = O.decode_step(params, dims, gpu_cache, past - 1, tok)
        assert rel_l2(got, ref_step) <= 1e-2
        top1_check(got, ref_step, 0.0, tie_tol=10 * float(np.sqrt(np.mean((got - ref_step) ** 2))))


def test_prefill_wide_batch_and_one_token_prompt():
    """B = 130 (> 128 rows: the lm_head writes logits and argmax_rows reads
    them) and a one-token prompt."""
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=1, n_pos=32, vocab=4000)
    params, d = synth.draw_model(dims, "bf16", 22)
    tokens = synth.draw_tokens(d, 130, 9, dims.vocab)
    _check_prefill(_Gen(dims, params, 130, 16), tokens, params, dims, seqs=(0, 77, 129))
    tokens = synth.draw_tokens(d, 2, 1, dims.vocab)
    _check_prefill(_Gen(dims, params, 2, 16), tokens, params, dims)


def test_prefill_argument_errors():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=1, n_pos=32, vocab=300)
    params, d = synth.draw_model(dims, "bf16", 2)
    g = _Gen(dims, params, 2, 16)
    ws = torch.empty(1 << 24, device="cuda", dtype=torch.uint8)
    tok = torch.zeros(2, 17, dtype=torch.int32, device="cuda")
    with pytest.raises(G.GPT2Error):  # T > T_max
        G.gpt2_prefill(g.cd, g.mw, tok, 2, 17, g.kv, 16, g.past, g.next, None, 0, ws, 1 << 24)
    with pytest.raises(G.GPT2Error):  # workspace too small
        G.gpt2_prefill(g.cd, g.mw, tok, 2, 8, g.kv, 16, g.past, g.next, None, 0, ws, 64)


def test_prefill_gpt2_small_b64_t1023():
    """The decode workload's prompt: B=64 sequences of 1023 tokens (GPT-2
    small, 1088 positions); the oracle checks sequence 0's cache of every
    layer and its last-position logits."""
    inp = synth.workload_inputs("gpt2_small_decode_b64")
    dims, params = inp["dims"], inp["params"]
    d = synth._Draw(4321, "bf16")
    tokens = synth.draw_tokens(d, 64, 1023, dims.vocab)
    g = _Gen(dims, params, 64, 1088)
    _check_prefill(g, tokens, params, dims, seqs=(0,))
    tok, _ = g.decode()
    assert np.array_equal(g.past.cpu().numpy(), np.full(64, 1024))
