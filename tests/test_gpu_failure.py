"""Failure detection on the GPU: a bounded wait that runs out.

Every mbarrier wait in the library's kernels gives up after a wall-time
limit, records GPT2_ERR_TIMEOUT with a site code in the device error word
and lets the kernel return, so that a producer that never delivers leaves
an error status instead of a hung GPU.  gpt2_selftest_wait_timeout runs that
same wait, in one GPU thread, on a barrier nothing ever arrives on, with a
short limit.  Nothing faults, traps or hangs: the test checks the status and
its site, that the wait lasted about its limit, and that the next ordinary
call on the same context succeeds.
"""
import numpy as np
import pytest

import oracle as O
from gpu_util import assert_close_elementwise, f32, rng, to_np, to_t

torch = pytest.importorskip("torch")
import gpt_pre_ln_gb300 as G  # noqa: E402

pytestmark = pytest.mark.gpu

SITE_SELFTEST_WAIT = 18


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gpt_pre_ln_gb300 import build
    build.build()
    G.lib()
    G.gpt2_last_error()  # start from a clear error word


def _layernorm_ok():
    r = rng(3)
    x = f32(r.standard_normal((40, 768)))
    g, b = f32(1 + 0.1 * r.standard_normal(768)), f32(0.1 * r.standard_normal(768))
    y = torch.empty(40, 768, device="cuda")
    G.gpt2_layernorm(to_t(x, "f32"), to_t(g, "f32"), to_t(b, "f32"), y, 40, 768, 1e-5, G.F32, G.F32)
    torch.cuda.synchronize()
    ref = O.layer_norm(x, g, b, 1e-5)
    assert_close_elementwise(to_np(y), ref, 1e-5 * np.abs(ref) + 1e-5, "layernorm after the timeout")


@pytest.mark.parametrize("limit_ms", [1.0, 20.0])
def test_wait_times_out_with_status_and_site(limit_ms):
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    G.gpt2_selftest_wait_timeout(int(limit_ms * 1e6))
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    st, site = G.gpt2_last_error()
    assert (st, site) == (5, SITE_SELFTEST_WAIT)
    assert 0.9 * limit_ms <= ms < limit_ms + 500.0, ms
    assert G.gpt2_last_error() == (0, 0)  # read once, then cleared
    _layernorm_ok()  # the context is still usable
    assert G.gpt2_last_error() == (0, 0)


def test_limit_outside_the_range_is_rejected():
    for bad in (0, 2_000_000_001):
        with pytest.raises(G.GPT2Error) as e:
            G.gpt2_selftest_wait_timeout(bad)
        assert e.value.status == 1
    assert G.gpt2_last_error() == (0, 0)
