"""The top-1 agreement a bf16 computation can reach, recomputed on the CPU.

The bf16 path's top-1 gate in the GPU parity tests is the flip rate of an
exact float64 forward that rounds only the tensor-core operands to bf16
(``bf16_emulation``).  This test recomputes that rate on the sampled
sequences of the GPT-2 small B=8, T=1024 workload, so the number behind the
gate is reproducible, and pins the emulation itself: with every rounding
removed it is the oracle, bit for bit; rounding in bf16 moves the logits by
the ~2^-9 relative step of the type (rel L2 a few 1e-3), not by more.
"""
import numpy as np
import pytest

import bf16_emulation as E
import oracle as O
import synth


def test_emulation_without_rounding_is_the_oracle(monkeypatch):
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2, vocab=500, n_pos=64)
    params, d = synth.draw_model(dims, "bf16", 31)
    tokens = synth.draw_tokens(d, 2, 40, dims.vocab)
    monkeypatch.setattr(E, "bf16", lambda a: np.asarray(a, np.float64))
    got = E.forward_logits_bf16_operands(tokens, params, dims)
    ref = O.forward_logits(tokens, params, dims)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_emulation_rounding_is_bf16_sized():
    dims = synth.replace_dims(synth.GPT2_SMALL, n_layer=2, vocab=500, n_pos=64)
    params, d = synth.draw_model(dims, "bf16", 32)
    tokens = synth.draw_tokens(d, 2, 40, dims.vocab)
    got = E.forward_logits_bf16_operands(tokens, params, dims)
    ref = O.forward_logits(tokens, params, dims)
    err = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert 2.0 ** -12 < err < 2.0 ** -6, err


def test_reachable_top1_agreement_on_the_sampled_workload():
    """98.975% (2027 of 2048 positions): below the 99.5% target for any
    bf16-operand computation on these weights."""
    agree, n, rel = E.agreement()
    print(f"bf16-operand emulation: top-1 agreement {agree}/{n} = {agree / n:.5f}, logits rel L2 {rel:.3e}")
    assert n == E.EMULATION_POSITIONS
    assert agree == E.EMULATION_AGREE
    assert rel == pytest.approx(E.EMULATION_REL_L2, rel=0.01)
