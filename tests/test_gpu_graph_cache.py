"""Repeated calls replayed as CUDA graphs.

On a stream other than the legacy default stream, the second call of a
multi-kernel entry point with the same arguments is captured into a CUDA
graph and every later one replays it.  A replay must give the bits of an
eager call (the same kernels with the same parameters), read the current
contents of every buffer (new token ids, changed weights at the same
addresses), and calls with different arguments must not replay another
call's graph.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
import gpt_pre_ln_gb300 as G  # noqa: E402

pytestmark = pytest.mark.gpu

DIMS = synth.Dims(n_layer=2, d_model=128, n_head=2, d_ff=512, vocab=1000, n_pos=256)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gpt_pre_ln_gb300 import build
    build.build()
    G.lib()
    yield
    st, site = G.gpt2_last_error()
    assert st == 0, f"device error {st} at site {site}"


def _model(seed):
    params, d = synth.draw_model(DIMS, "bf16", seed)
    dev = G.to_device(params, G.BF16)
    return params, d, dev


def _cd():
    return G.make_dims(DIMS.n_layer, DIMS.d_model, DIMS.n_head, DIMS.d_ff, DIMS.vocab, DIMS.n_pos, DIMS.eps, G.BF16)


def test_forward_logits_replay_matches_eager():
    params, d, dev = _model(31)
    mw, keep = G.model_weights(dev)
    cd = _cd()
    B, T = 2, 200
    ld = (DIMS.vocab + 7) // 8 * 8
    wsb = G.gpt2_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    tok_a = torch.from_numpy(synth.draw_tokens(d, B, T, DIMS.vocab)).cuda()
    tok_b = torch.from_numpy(synth.draw_tokens(d, B, T, DIMS.vocab)).cuda()

    def eager(tokens):  # the legacy default stream: always eager
        out = torch.full((B, T, ld), float("nan"), device="cuda")
        G.gpt2_forward_logits(cd, mw, tokens, out, ld, G.F32, B, T, ws, wsb, 0)
        torch.cuda.synchronize()
        return out

    ref_a, ref_b = eager(tok_a), eager(tok_b)
    side = torch.cuda.Stream()
    tok = tok_a.clone()
    out = torch.full((B, T, ld), float("nan"), device="cuda")
    for i in range(5):  # eager, captured, then replays
        src = tok_a if i % 2 == 0 else tok_b
        tok.copy_(src)
        torch.cuda.synchronize()
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        G.gpt2_forward_logits(cd, mw, tok, out, ld, G.F32, B, T, ws, wsb, side)
        side.synchronize()
        assert torch.equal(out[..., :DIMS.vocab], (ref_a if i % 2 == 0 else ref_b)[..., :DIMS.vocab]), i
    # weights changed in place: the replay reads the new values
    dev["blocks"][1]["w_fc"].mul_(-1.0)
    torch.cuda.synchronize()
    ref_c = eager(tok)
    G.gpt2_forward_logits(cd, mw, tok, out, ld, G.F32, B, T, ws, wsb, side)
    side.synchronize()
    assert torch.equal(out[..., :DIMS.vocab], ref_c[..., :DIMS.vocab])
    assert not torch.equal(ref_c, ref_a)  # (tok holds tok_a's ids)
    # another output buffer: another key, not the cached graph
    out2 = torch.full((B, T, ld), float("nan"), device="cuda")
    for _ in range(3):
        G.gpt2_forward_logits(cd, mw, tok, out2, ld, G.F32, B, T, ws, wsb, side)
    side.synchronize()
    assert torch.equal(out2[..., :DIMS.vocab], ref_c[..., :DIMS.vocab])
    del keep


def test_training_step_replay_matches_eager():
    params, d, dev = _model(32)
    mw, keep = G.model_weights(dev)
    cd = _cd()
    B, T = 2, 100
    tokens = torch.from_numpy(synth.draw_tokens(d, B, T, DIMS.vocab)).cuda()
    wsb = G.gpt2_train_workspace_bytes(cd, B, T)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)

    def grads():
        gd = {k: torch.full(tuple(dev[k].shape), float("nan"), device="cuda") for k in ("wte", "wpe", "lnf_g", "lnf_b")}
        gd["blocks"] = [{k: torch.full(tuple(v.shape), float("nan"), device="cuda") for k, v in b.items()}
                        for b in dev["blocks"]]
        return gd

    g0 = grads()
    mg0, k0 = G.model_grads(g0)
    loss0 = torch.full((1,), float("nan"), device="cuda")
    G.gpt2_forward_backward(cd, mw, tokens, None, mg0, loss0, B, T, ws, wsb, 0)
    torch.cuda.synchronize()
    g1 = grads()
    mg1, k1 = G.model_grads(g1)
    loss1 = torch.full((1,), float("nan"), device="cuda")
    side = torch.cuda.Stream()
    for _ in range(4):
        G.gpt2_forward_backward(cd, mw, tokens, None, mg1, loss1, B, T, ws, wsb, side)
    side.synchronize()
    assert torch.equal(loss0, loss1)
    assert torch.equal(g0["wte"], g1["wte"]) and torch.equal(g0["wpe"], g1["wpe"])
    for b0, b1 in zip(g0["blocks"], g1["blocks"]):
        for k in b0:
            assert torch.equal(b0[k], b1[k]), k
    del keep, k0, k1


def test_decode_steps_replay_match_eager():
    params, d, dev = _model(33)
    mw, keep = G.model_weights(dev)
    cd = _cd()
    B, T0, T_max, steps = 3, 40, 64, 5
    prompt = torch.from_numpy(synth.draw_tokens(d, B, T0, DIMS.vocab)).cuda()
    kvb = G.gpt2_kv_cache_bytes(cd, B, T_max)
    wsb_p = G.gpt2_prefill_workspace_bytes(cd, B, T0)
    wsb_d = G.gpt2_decode_workspace_bytes(cd, B)

    def run(stream, sync):
        kv = torch.zeros(kvb, device="cuda", dtype=torch.uint8)
        past = torch.zeros(B, device="cuda", dtype=torch.int32)
        nxt = torch.zeros(B, device="cuda", dtype=torch.int32)
        ws_p = torch.empty(wsb_p, device="cuda", dtype=torch.uint8)
        ws_d = torch.empty(wsb_d, device="cuda", dtype=torch.uint8)
        G.gpt2_prefill(cd, mw, prompt, B, T0, kv, T_max, past, nxt, None, 0, ws_p, wsb_p, 0)
        torch.cuda.synchronize()
        tok = nxt.clone()
        seq = []
        for _ in range(steps):
            G.gpt2_decode_step(cd, mw, kv, B, T_max, past, tok, nxt, None, 0, ws_d, wsb_d, stream)
            sync()
            torch.cuda.synchronize()
            seq.append(nxt.cpu().numpy().copy())
            tok.copy_(nxt)
            torch.cuda.synchronize()
        return np.stack(seq), kv, past

    s_eager, kv_e, past_e = run(0, torch.cuda.synchronize)
    side = torch.cuda.Stream()
    s_graph, kv_g, past_g = run(side, side.synchronize)
    np.testing.assert_array_equal(s_eager, s_graph)
    assert torch.equal(past_e, past_g) and torch.equal(kv_e, kv_g)
    del keep
