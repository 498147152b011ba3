"""Helpers shared by the GPU parity tests (inputs, tolerances, metrics)."""
from __future__ import annotations

import numpy as np

import synth


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def bf16(a):
    return synth.round_to(a, "bf16")


def f32(a):
    return synth.round_to(a, "f32")


def f16(a):
    return synth.round_to(a, "f16")


def to_t(a, dtype, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}.get(dtype, torch.float32)
    return t.to(tdt).contiguous()


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def max_rel_err(got, ref):
    """max_i |g - r| / max(|r_i|, rms(r)): relative error that does not blow
    up on entries near zero (the fp32 gate's definition)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), rms)))


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def assert_close_elementwise(got, ref, bound, what=""):
    """Every |got - ref| <= bound (arrays broadcast)."""
    err = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} entries out of bound; first at {tuple(idx)}: "
                             f"got {np.asarray(got)[tuple(idx)]}, ref {np.asarray(ref)[tuple(idx)]}, "
                             f"bound {np.broadcast_to(bound, err.shape)[tuple(idx)]}")


def top1_check(got_logits, ref_logits, min_agree=0.995, tie_tol=None):
    """Top-1 agreement rate, and every disagreement must be a near tie: the
    oracle's score of the GPU's choice is within ``tie_tol`` of the oracle's
    maximum (several answers are then correct within the error bound)."""
    g = np.argmax(got_logits, -1)
    r = np.argmax(ref_logits, -1)
    agree = float(np.mean(g == r))
    if tie_tol is not None:
        ref_at_g = np.take_along_axis(ref_logits, g[..., None], -1)[..., 0]
        gap = ref_logits.max(-1) - ref_at_g
        assert np.all(gap <= tie_tol), f"a flipped argmax is not a near tie (gap {gap.max()} > {tie_tol})"
    assert agree >= min_agree, f"top-1 agreement {agree:.4f} < {min_agree}"
    return agree
