"""Block, whole-forward and decode-step parity on the GPU against the oracle.

Gates (the accuracy targets of this path, restated here):
* F32 path, one block: max relative error <= 1e-4 on the hidden state, with
  the error measured as max_i |g - r| / max(|r_i|, rms(r)).
* BF16 path, logits: relative L2 <= 1e-2, and every argmax that differs
  must be a near tie in the oracle's own scores.  Top-1 agreement is held to
  the flip rate of an exact computation that rounds the GEMM inputs to bf16
  (about 1%, with a binomial allowance for the sample size): the 99.5% target
  is out of reach for any such computation at these random-init weights.
* BF16 path, one block's hidden state: relative L2 <= 2e-3.  A single block
  at random init changes the residual stream by ~5-10%; a dropped bias or a
  dropped sublayer would move it by ~1e-2, so the gate sits below that.
"""
import numpy as np
import pytest

import oracle as O
import synth
from bf16_emulation import EMULATION_AGREE, EMULATION_POSITIONS, SAMPLED_SEQUENCES
from gpu_util import max_rel_err, rel_l2, rng, to_np, to_t, top1_check

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


def _dims(d: synth.Dims, dtype):
    return G.make_dims(d.n_layer, d.d_model, d.n_head, d.d_ff, d.vocab, d.n_pos, d.eps,
                       G.BF16 if dtype == "bf16" else G.F32)


def _run_block(inp, B, T):
    dims = inp["dims"]
    dt = G.BF16 if inp["dtype"] == "bf16" else G.F32
    dev = G.to_device(inp["params"], dt)
    cd = _dims(dims, inp["dtype"])
    bw = G.block_weights(dev["blocks"][0])
    x = to_t(inp["x"], "f32")
    out = torch.empty_like(x)
    wsb = G.gpt2_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_block_forward(cd, bw, x, out, B, T, ws, wsb)
    torch.cuda.synchronize()
    return to_np(out)


def test_block_fp32_config0():
    """One GPT-2 small block in fp32, B=1, T=64, X ~ N(0, 1)."""
    inp = synth.workload_inputs("block_fp32_b1_t64")
    got = _run_block(inp, 1, 64)
    p = inp["params"]["blocks"][0]
    ref = O.block_forward(inp["x"], p, inp["dims"].n_head, inp["dims"].eps)
    err = max_rel_err(got, ref)
    assert err <= 1e-4, err
    assert rel_l2(ref, inp["x"]) > 1e-2  # the block changed the state


@pytest.mark.parametrize("B,T", [(2, 37), (1, 129)])
def test_block_fp32_ragged(B, T):
    inp = synth.workload_inputs("block_fp32_b1_t64", T_override=T, B_override=B)
    got = _run_block(inp, B, T)
    ref = O.block_forward(inp["x"], inp["params"]["blocks"][0], 12, 1e-5)
    assert max_rel_err(got, ref) <= 1e-4


@pytest.mark.parametrize("B,T", [(2, 200), (1, 1024)])
def test_block_bf16(B, T):
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=1)
    params, d = synth.draw_model(dims, "bf16", 4321, with_embeddings=False)
    x = synth.draw_activations(d, B, T, dims.d_model)
    inp = {"dims": dims, "dtype": "bf16", "params": params, "x": x}
    got = _run_block(inp, B, T)
    ref = O.block_forward(x, params["blocks"][0], 12, 1e-5)
    assert rel_l2(got, ref) <= 2e-3, rel_l2(got, ref)
    assert rel_l2(ref, x) > 2e-2


def test_block_in_place():
    inp = synth.workload_inputs("block_fp32_b1_t64")
    dev = G.to_device(inp["params"], G.F32)
    cd = _dims(inp["dims"], "f32")
    x = to_t(inp["x"], "f32")
    wsb = G.gpt2_workspace_bytes(cd, 1, 64)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_block_forward(cd, G.block_weights(dev["blocks"][0]), x, x, 1, 64, ws, wsb)
    torch.cuda.synchronize()
    ref = O.block_forward(inp["x"], inp["params"]["blocks"][0], 12, 1e-5)
    assert max_rel_err(to_np(x), ref) <= 1e-4


def _forward(dims, dtype, params, tokens, logits_t=G.BF16):
    B, T = tokens.shape
    dev = G.to_device(params, G.BF16 if dtype == "bf16" else G.F32)
    mw, keep = G.model_weights(dev)
    cd = _dims(dims, dtype)
    ld = (dims.vocab + 7) // 8 * 8
    logits = torch.empty(B, T, ld, device="cuda", dtype=torch.bfloat16 if logits_t == G.BF16 else torch.float32)
    wsb = G.gpt2_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    tok = torch.from_numpy(tokens).to("cuda")
    G.gpt2_forward_logits(cd, mw, tok, logits, ld, logits_t, B, T, ws, wsb)
    torch.cuda.synchronize()
    del keep
    return logits[..., :dims.vocab]


# Top-1 agreement reachable by a path that rounds the GEMM inputs (LayerNorm
# outputs, QKV, probabilities, attention output, MLP hidden) to bf16: an
# exact float64 computation with only those roundings (bf16_emulation,
# recomputed by test_bf16_emulation.py) agrees with the oracle on 2027 of the
# 2048 positions of the two sampled GPT-2 small sequences (98.975%, rel L2
# 3.85e-3), because random-init logits have top-1/top-2 gaps down to 1e-4.
# The bf16 path is held to that flip rate with a 3-sigma binomial allowance
# for the number of positions checked; every flip must be a near tie.
BF16_PATH_FLIP_RATE = 1.0 - EMULATION_AGREE / EMULATION_POSITIONS


def _min_top1(n):
    p = BF16_PATH_FLIP_RATE
    allowed = n * p + 3.0 * np.sqrt(n * p * (1.0 - p)) + 1.0
    return 1.0 - allowed / n


def _check_logits(got, ref, fp32_logits=True):
    """rel L2 <= 1e-2; with fp32 logits, top-1 agreement within the bf16
    path's flip rate (see above); every differing argmax a near tie.

    bf16 logits are rounded to 8 significant bits (a step of 2^-6 near the
    largest scores), which creates exact ties and flips far more often than
    the arithmetic before the rounding does; for them only the near-tie
    check applies.
    """
    err = rel_l2(got, ref)
    rms_err = float(np.sqrt(np.mean((got - ref) ** 2)))
    n = int(np.prod(got.shape[:-1]))
    agree = float(np.mean(np.argmax(got, -1) == np.argmax(ref, -1)))
    print(f"logits rel L2 {err:.3e}, rms err {rms_err:.3e}, top-1 agreement {agree:.5f} over {n}")
    assert err <= 1e-2, err
    top1_check(got, ref, _min_top1(n) if fp32_logits else 0.0, tie_tol=10 * rms_err)
    return err


@pytest.mark.parametrize("logits_t", [G.BF16, G.F32])
def test_forward_logits_small_stack(logits_t):
    """Two GPT-2-small-width blocks, full vocabulary, ragged T."""
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2)
    params, d = synth.draw_model(dims, "bf16", 99)
    tokens = synth.draw_tokens(d, 2, 150, dims.vocab)
    got = to_np(_forward(dims, "bf16", params, tokens, logits_t))
    ref = O.forward_logits(tokens, params, dims)
    _check_logits(got, ref, fp32_logits=logits_t == G.F32)


def test_forward_logits_fp32_path():
    dims = synth.Dims(n_layer=2, d_model=128, n_head=2, d_ff=512, vocab=1000, n_pos=64)
    params, d = synth.draw_model(dims, "f32", 7)
    tokens = synth.draw_tokens(d, 2, 50, dims.vocab)
    got = to_np(_forward(dims, "f32", params, tokens, G.F32))
    ref = O.forward_logits(tokens, params, dims)
    assert max_rel_err(got, ref) <= 1e-4


def test_forward_logits_causality():
    """Changing later tokens leaves the logits of earlier positions bit-identical."""
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2, vocab=5000)
    params, d = synth.draw_model(dims, "bf16", 5)
    tokens = synth.draw_tokens(d, 1, 256, dims.vocab)
    a = _forward(dims, "bf16", params, tokens)
    t2 = tokens.copy()
    t2[0, 100:] = (t2[0, 100:] + 17) % dims.vocab
    b = _forward(dims, "bf16", params, t2)
    # rows 0..99 share every input they may depend on
    assert torch.equal(a[:, :100], b[:, :100])
    assert not torch.equal(a[:, 100:], b[:, 100:])


def test_forward_logits_gpt2_small_full_size():
    """GPT-2 small, B=8, T=1024 (the benchmark's launch configuration).

    The GPU runs the whole batch; the oracle checks two sampled sequences.
    """
    inp = synth.workload_inputs("gpt2_small_fwd_b8_t1024")
    dims, params, tokens = inp["dims"], inp["params"], inp["tokens"]
    logits = _forward(dims, "bf16", params, tokens, G.F32)
    got = np.concatenate([to_np(logits[b:b + 1]) for b in SAMPLED_SEQUENCES])
    ref = np.concatenate([O.forward_logits(tokens[b:b + 1], params, dims) for b in SAMPLED_SEQUENCES])
    # the positions the emulation's agreement was counted on, pooled
    _check_logits(got, ref)


@pytest.mark.parametrize("name,seqs", [("gpt2_medium_fwd_b16_t1024", (15,)), ("gpt2_xl_fwd_b4_t1024", (3,))],
                         ids=["gpt2-medium-b16", "gpt2-xl-b4"])
def test_forward_logits_larger_models_full_size(name, seqs):
    """GPT-2 medium (24 x 1024, 16 heads; B=16) and XL (48 x 1600, 25 heads;
    B=4) at T=1024: the GPU runs the whole batch, the oracle checks the last
    sequence at every position."""
    inp = synth.workload_inputs(name)
    dims, params, tokens = inp["dims"], inp["params"], inp["tokens"]
    logits = _forward(dims, "bf16", params, tokens, G.F32)
    for b in seqs:
        got = to_np(logits[b:b + 1])
        ref = O.forward_logits(tokens[b:b + 1], params, dims)
        _check_logits(got, ref)


def test_embedding_token_out_of_range_is_reported():
    dims = synth.Dims(n_layer=1, d_model=128, n_head=2, d_ff=512, vocab=100, n_pos=16)
    params, _ = synth.draw_model(dims, "bf16", 1)
    tokens = np.array([[1, 2, 100, 3]], dtype=np.int32)
    _forward(dims, "bf16", params, tokens)
    st, site = G.gpt2_last_error()
    assert st == 6 and site == 10
    assert G.gpt2_last_error()[0] == 0  # cleared after reading


# --------------------------------------------------------------------- decode
def _decode_setup(dims, B, T_max, past, seed):
    params, d = synth.draw_model(dims, "bf16", seed)
    cache = np.zeros((dims.n_layer, 2, B, dims.n_head, T_max, 64), np.float32)
    for b in range(B):
        cache[:, :, b, :, :past[b]] = synth.round_to(
            d.rng.standard_normal((dims.n_layer, 2, dims.n_head, past[b], 64)), "bf16")
    tokens = d.rng.integers(0, dims.vocab, size=B).astype(np.int32)
    return params, cache, tokens


def test_decode_steps_match_oracle():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2, n_pos=64)
    B, T_max = 3, 48
    past = np.array([5, 40, 17], np.int32)
    params, cache, tokens = _decode_setup(dims, B, T_max, past, 11)
    dev = G.to_device(params, G.BF16)
    mw, keep = G.model_weights(dev)
    cd = _dims(dims, "bf16")
    kv = to_t(cache, "bf16")
    pl = torch.from_numpy(past.copy()).to("cuda")
    tok = torch.from_numpy(tokens.copy()).to("cuda")
    nxt = torch.empty_like(tok)
    ld = 50264
    logits = torch.empty(B, ld, device="cuda")
    wsb = G.gpt2_decode_workspace_bytes(cd, B)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    ocache, opast, otok = cache.astype(np.float64), past.copy(), tokens.copy()
    for step in range(4):
        G.gpt2_decode_step(cd, mw, kv, B, T_max, pl, tok, nxt, logits, ld, ws, wsb)
        torch.cuda.synchronize()
        _, ref_logits, ocache, opast = O.decode_step(params, dims, ocache, opast, otok)
        got = to_np(logits[:, :dims.vocab])
        _check_logits(got, ref_logits)
        assert np.array_equal(pl.cpu().numpy(), opast)
        g_next = nxt.cpu().numpy()
        assert np.array_equal(g_next, np.argmax(got, -1))  # the kernel's argmax of its own logits
        otok = g_next  # both sides continue from the GPU's choice
        tok.copy_(nxt)
    # the cache slots written by the GPU hold the new k, v of the oracle (up
    # to the bf16 rounding of the c_attn input and output: ~3e-3 relative;
    # a value in the wrong slot or head would be off by ~100%)
    kv_np = to_np(kv)
    for b in range(B):
        for s in range(past[b], past[b] + 4):
            for l in range(dims.n_layer):
                for kvi in range(2):
                    assert rel_l2(kv_np[l, kvi, b, :, s], ocache[l, kvi, b, :, s]) < 2e-2, (b, s, l, kvi)
        assert np.all(kv_np[:, :, b, :, past[b] + 4:] == 0)
        np.testing.assert_array_equal(kv_np[:, :, b, :, :past[b]], ocache[:, :, b, :, :past[b]])
    del keep


def test_decode_position_out_of_range_is_reported():
    dims = synth.Dims(n_layer=1, d_model=128, n_head=2, d_ff=512, vocab=50, n_pos=16)
    B, T_max = 2, 8
    past = np.array([3, 8], np.int32)  # the second sequence's cache is full
    params, cache, tokens = _decode_setup(dims, B, T_max, np.array([3, 8]), 2)
    dev = G.to_device(params, G.BF16)
    mw, keep = G.model_weights(dev)
    cd = _dims(dims, "bf16")
    kv = to_t(cache, "bf16")
    pl = torch.from_numpy(past.copy()).to("cuda")
    tok = torch.from_numpy(tokens.copy()).to("cuda")
    nxt = torch.full_like(tok, -7)
    wsb = G.gpt2_decode_workspace_bytes(cd, B)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_decode_step(cd, mw, kv, B, T_max, pl, tok, nxt, None, 0, ws, wsb)
    st, site = G.gpt2_last_error()
    assert st == 6 and site == 11
    assert pl.cpu().tolist() == [4, 8]
    assert nxt.cpu().tolist()[1] == -7 and nxt.cpu().tolist()[0] >= 0
    del keep


@pytest.mark.parametrize("B", [20, 130])
def test_decode_batches(B):
    """Sequences with mixed cache lengths.  At B = 130 the batch is past the
    few-row GEMM (128 rows), so the lm_head writes fp32 logits and a separate
    kernel takes the argmax; below, the lm_head's epilogue makes argmax
    candidates.  Both must pick the argmax of the step's own logits and
    match the oracle."""
    dims = synth.Dims(n_layer=2, d_model=128, n_head=2, d_ff=512, vocab=300, n_pos=16)
    T_max = 8
    past = (np.arange(B) % 7).astype(np.int32)
    params, cache, tokens = _decode_setup(dims, B, T_max, past, 3)
    dev = G.to_device(params, G.BF16)
    mw, keep = G.model_weights(dev)
    cd = _dims(dims, "bf16")
    kv = to_t(cache, "bf16")
    pl = torch.from_numpy(past.copy()).to("cuda")
    tok = torch.from_numpy(tokens.copy()).to("cuda")
    nxt = torch.empty_like(tok)
    ld = 304
    logits = torch.empty(B, ld, device="cuda")
    wsb = G.gpt2_decode_workspace_bytes(cd, B)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_decode_step(cd, mw, kv, B, T_max, pl, tok, nxt, logits, ld, ws, wsb)
    torch.cuda.synchronize()
    got = to_np(logits[:, :dims.vocab])
    _, ref, ocache, opast = O.decode_step(params, dims, cache.astype(np.float64), past.copy(), tokens.copy())
    _check_logits(got, ref)
    assert np.array_equal(nxt.cpu().numpy(), np.argmax(got, -1))
    assert np.array_equal(pl.cpu().numpy(), opast)
    kv_np = to_np(kv)
    for b in range(B):  # the new slot of every sequence, in its own cache rows
        s_ = past[b]
        assert rel_l2(kv_np[:, :, b, :, s_], ocache[:, :, b, :, s_]) < 2e-2, b
        assert np.all(kv_np[:, :, b, :, s_ + 1:] == 0)
    del keep
