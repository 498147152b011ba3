"""Decode steps at the decode workload's context lengths, against the oracle.

The decode attention splits each sequence's cached keys into 16-key chunks
that four warps per (sequence, head) stream through two-slot rings, so a
context of n keys makes each warp's ring wrap about n / 128 times.  These
tests reach every case of that walk ("逐行拆GPT-2源码", GPT2Attention: the
new K and V are appended to the cached ones along the sequence axis, and
GPT2Model: positions continue from past_length):

* a one-layer model (D = 128, two heads) decoded with past lengths 0, 1, 15,
  16, 17, 63, 64, 65, 127, 128, 129, 511, 1023 and 1086 in one batch, two
  steps;
* the decode workload itself: GPT-2 small, B = 64, 1023 cached positions
  per sequence (1088 position rows), six greedy steps, with the oracle
  following three of the sequences.

Gates (those of the other decode tests): logits rel L2 <= 1e-2 per step;
the token chosen is the argmax of the step's own logits, and the oracle's
argmax or a near tie in the oracle's scores; each K/V slot the step writes
within 2e-2 rel L2 of the oracle's (bf16 rounding of the c_attn input and
output: ~3e-3; a row in the wrong slot or head is off by ~100%); cached
slots untouched bit for bit, slots beyond the new ones still zero.
"""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_util import rel_l2, to_np, to_t, top1_check

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


def _cd(dims):
    return G.make_dims(dims.n_layer, dims.d_model, dims.n_head, dims.d_ff, dims.vocab, dims.n_pos, dims.eps, G.BF16)


def _check_step(got_logits, ref_logits, got_next):
    assert rel_l2(got_logits, ref_logits) <= 1e-2, rel_l2(got_logits, ref_logits)
    assert np.array_equal(got_next, np.argmax(got_logits, -1))
    rms = float(np.sqrt(np.mean((got_logits - ref_logits) ** 2)))
    top1_check(got_logits, ref_logits, 0.0, tie_tol=10 * rms)


PAST_LENS = [0, 1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 511, 1023, 1086]


def test_decode_every_ring_phase():
    dims = synth.Dims(n_layer=1, d_model=128, n_head=2, d_ff=512, vocab=1000, n_pos=1088)
    B, T_max = len(PAST_LENS), 1088
    past = np.array(PAST_LENS, np.int32)
    params, d = synth.draw_model(dims, "bf16", 1601)
    cache = np.zeros((1, 2, B, dims.n_head, T_max, 64), np.float32)
    for b in range(B):
        cache[:, :, b, :, :past[b]] = synth.round_to(d.rng.standard_normal((1, 2, dims.n_head, past[b], 64)), "bf16")
    tokens = d.rng.integers(0, dims.vocab, size=B).astype(np.int32)
    dev = G.to_device(params, G.BF16)
    mw, keep = G.model_weights(dev)
    cd = _cd(dims)
    kv = to_t(cache, "bf16")
    pl = torch.from_numpy(past.copy()).cuda()
    tok = torch.from_numpy(tokens.copy()).cuda()
    nxt = torch.empty_like(tok)
    ld = 1000
    logits = torch.empty(B, ld, device="cuda")
    wsb = G.gpt2_decode_workspace_bytes(cd, B)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    ocache, opast, otok = cache.astype(np.float64), past.copy(), tokens.copy()
    steps = 2
    for _ in range(steps):
        G.gpt2_decode_step(cd, mw, kv, B, T_max, pl, tok, nxt, logits, ld, ws, wsb)
        torch.cuda.synchronize()
        _, ref, ocache, opast = O.decode_step(params, dims, ocache, opast, otok)
        got = to_np(logits)
        g_next = nxt.cpu().numpy()
        _check_step(got, ref, g_next)
        # per sequence too: every context length must be right on its own
        for b in range(B):
            assert rel_l2(got[b], ref[b]) <= 1e-2, (PAST_LENS[b], rel_l2(got[b], ref[b]))
        assert np.array_equal(pl.cpu().numpy(), opast)
        otok = g_next
        tok.copy_(nxt)
    kv_np = to_np(kv)
    for b in range(B):
        p = past[b]
        for s in range(p, p + steps):
            for kvi in range(2):
                assert rel_l2(kv_np[0, kvi, b, :, s], ocache[0, kvi, b, :, s]) < 2e-2, (p, s, kvi)
        np.testing.assert_array_equal(kv_np[:, :, b, :, :p], cache[:, :, b, :, :p])
        assert np.all(kv_np[:, :, b, :, p + steps:] == 0)
    assert G.gpt2_last_error() == (0, 0)
    del keep


SAMPLED = (0, 31, 63)


def test_decode_workload_full_size():
    """GPT-2 small, B = 64, 1023 cached positions, six greedy steps: the GPU
    runs the whole batch, the oracle follows sequences 0, 31 and 63."""
    inp = synth.workload_inputs("gpt2_small_decode_b64", cache_as_slabs=True)
    dims, params, tokens = inp["dims"], inp["params"], inp["tokens"]
    B, T_max, fill = inp["B"], inp["T_max"], inp["workload"].cache_len
    L, H = dims.n_layer, dims.n_head
    kv = torch.zeros(L, 2, B, H, T_max, 64, dtype=torch.bfloat16, device="cuda")
    ocache = np.zeros((L, 2, len(SAMPLED), H, T_max, 64))
    for l, kvi, slab in inp["cache_slabs"]:
        kv[l, kvi, :, :, :fill] = torch.from_numpy(slab).cuda().to(torch.bfloat16)
        ocache[l, kvi, :, :, :fill] = slab[list(SAMPLED)]
    dev = G.to_device(params, G.BF16)
    mw, keep = G.model_weights(dev)
    cd = _cd(dims)
    pl = torch.from_numpy(inp["past_len"].copy()).cuda()
    tok = torch.from_numpy(tokens.copy()).cuda()
    nxt = torch.empty_like(tok)
    ld = (dims.vocab + 3) // 4 * 4
    logits = torch.empty(B, ld, device="cuda")
    wsb = G.gpt2_decode_workspace_bytes(cd, B)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    opast = np.full(len(SAMPLED), fill, np.int32)
    otok = tokens[list(SAMPLED)].copy()
    steps = 6
    for step in range(steps):
        G.gpt2_decode_step(cd, mw, kv, B, T_max, pl, tok, nxt, logits, ld, ws, wsb)
        torch.cuda.synchronize()
        _, ref, ocache, opast = O.decode_step(params, dims, ocache, opast, otok)
        got = to_np(logits[list(SAMPLED), :dims.vocab])
        g_next_all = nxt.cpu().numpy()
        g_next = g_next_all[list(SAMPLED)]
        _check_step(got, ref, g_next)
        assert np.all((g_next_all >= 0) & (g_next_all < dims.vocab))
        assert np.array_equal(pl.cpu().numpy(), np.full(B, fill + step + 1))
        otok = g_next
        tok.copy_(nxt)
    for i, b in enumerate(SAMPLED):
        kb = kv[:, :, b].float().cpu().numpy()  # [L, 2, H, T_max, 64]
        for s in range(fill, fill + steps):
            for l in range(L):
                for kvi in range(2):
                    assert rel_l2(kb[l, kvi, :, s], ocache[l, kvi, i, :, s]) < 2e-2, (b, s, l, kvi)
        np.testing.assert_array_equal(kb[:, :, :, :fill], ocache[:, :, i, :, :fill])
        assert np.all(kb[:, :, :, fill + steps:] == 0)
    assert G.gpt2_last_error() == (0, 0)
    del keep
