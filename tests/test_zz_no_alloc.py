"""gpt2_mlp_noalloc: the MLP entry point for callers that cannot allocate.

Some callers cannot allocate device memory at the moment they call the MLP
(a plug-in inside a framework that owns the GPU's memory pool, code running
during CUDA graph capture).  gpt2_mlp_noalloc takes the same arguments as
gpt2_mlp minus the workspace and keeps the hidden activation in a fixed
scratch array owned by the library.  Both entry points issue the same two
GEMM launches on the same inputs, so their outputs must agree bit for bit;
this test calls both through the C ABI and checks that, on two calls in a
row (the array keeps the previous call's contents), checks the first call
against the float64 oracle within the MLP parity test's bound, and checks
the size limit.  The file sorts last so that a run stopping at the first
failure has run every other test before it.
"""
import numpy as np
import pytest

import oracle as O
from gpu_util import assert_close_elementwise, bf16, f32, rng, to_np, to_t

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


def _inputs(seed, M, D, F):
    r = rng(seed)
    x = bf16(r.standard_normal((M, D)))
    w_fc, b_fc = bf16(0.02 * r.standard_normal((D, F))), bf16(0.01 * r.standard_normal(F))
    w_p, b_p = bf16(0.004 * r.standard_normal((F, D))), bf16(0.01 * r.standard_normal(D))
    res = f32(r.standard_normal((M, D)))
    return x, w_fc, b_fc, w_p, b_p, res


@pytest.mark.parametrize("with_res", [True, False])
def test_noalloc_matches_workspace_entry_point_twice(with_res):
    M, D, F = 300, 768, 3072
    for call, seed in enumerate((41, 42)):  # two calls in a row, different inputs
        arrays = _inputs(seed, M, D, F)
        x, w_fc, b_fc, w_p, b_p, res = (to_t(a, "bf16" if i < 5 else "f32") for i, a in enumerate(arrays))
        ref = torch.empty(M, D, device="cuda")
        got = torch.full((M, D), float("nan"), device="cuda")
        wsb = G.gpt2_mlp_workspace_bytes(M, F, G.BF16)
        ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
        G.gpt2_mlp(x, w_fc, b_fc, w_p, b_p, res if with_res else None, ref, M, D, F, ws, wsb, G.BF16)
        G.gpt2_mlp_noalloc(x, w_fc, b_fc, w_p, b_p, res if with_res else None, got, M, D, F, G.BF16)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {call}: the two entry points differ"
        if call == 0:
            # anchored to the oracle with the MLP parity test's bound: the
            # hidden activation is rounded to bf16 (2^-9 relative) before c_proj
            xa, wf, bf, wp, bp, ra = arrays
            blk = {"w_fc": wf, "b_fc": bf, "w_proj": wp, "b_proj": bp}
            o_ref = O.mlp_forward(xa, blk) + (ra if with_res else 0)
            g_abs = np.abs(O.gelu_new(xa @ wf.astype(np.float64) + bf))
            bound = 2.0 ** -8 * (g_abs @ np.abs(wp.astype(np.float64))) + 2.0 ** -20 * np.abs(o_ref) + 1e-6
            assert_close_elementwise(to_np(got), o_ref, bound, "noalloc against the oracle")


def test_noalloc_fp32_path():
    M, D, F = 70, 128, 512
    x, w_fc, b_fc, w_p, b_p, res = _inputs(7, M, D, F)
    t = [to_t(a, "f32") for a in (x, w_fc, b_fc, w_p, b_p, res)]
    ref = torch.empty(M, D, device="cuda")
    got = torch.empty(M, D, device="cuda")
    wsb = G.gpt2_mlp_workspace_bytes(M, F, G.F32)
    ws = torch.empty(wsb, device="cuda", dtype=torch.uint8)
    G.gpt2_mlp(*t[:5], t[5], ref, M, D, F, ws, wsb, G.F32)
    G.gpt2_mlp_noalloc(*t[:5], t[5], got, M, D, F, G.F32)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


def test_noalloc_rejects_sizes_beyond_the_scratch():
    cap = G.gpt2_mlp_noalloc_max_scratch_bytes()
    assert cap == 16 << 20
    F = 3072
    M = cap // (F * 2) + 1  # one row more than fits
    dummy = torch.empty(64, device="cuda")
    with pytest.raises(G.GPT2Error) as e:
        G.gpt2_mlp_noalloc(dummy, dummy, dummy, dummy, dummy, None, dummy, M, 768, F, G.BF16)
    assert e.value.status == 3
