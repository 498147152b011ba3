"""Host-side checks of the C ABI that need no GPU.

The library must load on a machine without a GPU driver, export every
function that include/gpt2gb.h declares, agree with the header's constants,
and reject bad arguments before anything reaches the device.  No call here
launches GPU work.
"""
import ctypes
import os
import re

import pytest

import gpt_pre_ln_gb300 as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gpt2gb.h")


@pytest.fixture(scope="module")
def L():
    from gpt_pre_ln_gb300 import build
    build.build()
    return G.lib()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gpt2_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for n in ("gpt2_layernorm", "gpt2_attention_causal", "gpt2_mlp", "gpt2_block_forward", "gpt2_forward_logits",
              "gpt2_decode_step", "gpt2_workspace_bytes", "gpt2_kv_cache_bytes", "gpt2_last_error",
              "gpt2_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared_functions():
        assert hasattr(L, n), n
        assert n in G._SIGS, f"binding lacks a signature for {n}"


def test_header_constants_match_binding():
    src = open(HEADER).read()
    consts = dict((k, int(v)) for k, v in re.findall(r"\b(GPT2_[A-Z0-9_]+)\s*=\s*(\d+)", src))
    assert consts["GPT2_F32"] == G.F32 and consts["GPT2_BF16"] == G.BF16
    assert consts["GPT2_EPI_BIAS_GELU"] == G.EPI_BIAS_GELU and consts["GPT2_EPI_BIAS_RESIDUAL"] == G.EPI_BIAS_RESIDUAL
    assert consts["GPT2_W_OUT_IN"] == G.W_OUT_IN
    assert consts["GPT2_ERR_TIMEOUT"] == 5 and consts["GPT2_ERR_RANGE"] == 6
    assert consts["GPT2_EPI_BIAS_GELU_EXACT"] == G.EPI_BIAS_GELU_EXACT
    assert consts["GPT2_SCALE_ATTN_BY_INVERSE_LAYER_IDX"] == G.SCALE_ATTN_BY_INVERSE_LAYER_IDX
    assert consts["GPT2_GELU_EXACT"] == G.GELU_EXACT


def test_struct_layout_matches_header(L):
    assert ctypes.sizeof(G.Dims) == 9 * 4
    assert ctypes.sizeof(G.BlockWeights) == 12 * 8
    assert ctypes.sizeof(G.ModelWeights) == 5 * 8


def test_status_strings(L):
    assert G.gpt2_abi_version() == 4
    assert G.gpt2_status_string(0) == "ok"
    assert "workspace" in G.gpt2_status_string(3)


def test_workspace_queries(L):
    d = G.make_dims(12, 768, 12, 3072, 50257, 1024)
    M = 8 * 1024
    ws = G.gpt2_workspace_bytes(d, 8, 1024)
    expect = 2 * M * 768 * 4 + 2 * M * 768 * 2 + M * 3 * 768 * 2 + M * 3072 * 2
    assert ws == expect
    assert G.gpt2_kv_cache_bytes(d, 64, 1087) == 12 * 2 * 64 * 12 * 1087 * 64 * 2
    assert G.gpt2_mlp_workspace_bytes(100, 3072, G.BF16) == ((100 * 3072 * 2 + 255) // 256) * 256
    assert G.gpt2_decode_workspace_bytes(d, 64) > 0
    bad = G.make_dims(12, 768, 10, 3072, 50257, 1024)  # head_dim not 64
    assert G.gpt2_workspace_bytes(bad, 8, 1024) == 0


def test_argument_checks_before_any_launch(L):
    """Calls with bad arguments return an error status without touching the GPU."""
    assert L.gpt2_layernorm(None, None, None, None, 10, 768, 1e-5, 0, 7, None) == 1       # bad dtype
    assert L.gpt2_layernorm(16, 16, 16, 16, 10, 770, 1e-5, 0, 0, None) == 2             # D % 4
    assert L.gpt2_layernorm(16, 16, 16, 16, -1, 768, 1e-5, 0, 0, None) == 1             # rows < 0
    assert L.gpt2_layernorm(16, 16, 16, 16, 10, 768, 0.0, 0, 0, None) == 1              # eps <= 0
    assert L.gpt2_layernorm(0, 0, 0, 0, 0, 768, 1e-5, 0, 0, None) == 0                  # empty: no-op
    assert L.gpt2_linear(16, 16, 16, None, 16, 10, 768, 700, 768, 0, 1, 1, 1, None) == 2  # K % 64
    assert L.gpt2_linear(16, 16, 16, None, 16, 10, 768, 768, 700, 0, 1, 1, 1, None) == 1  # ldy < N
    assert L.gpt2_linear(16, 16, 16, None, 16, 10, 768, 768, 768, 0, 3, 1, 1, None) == 2  # residual needs fp32 y
    assert L.gpt2_linear(16, 16, None, None, 16, 10, 768, 768, 768, 0, 1, 1, 1, None) == 1  # bias missing
    assert L.gpt2_linear(16, 16, 16, None, 16, 10, 770, 768, 770, 0, 1, 1, 1, None) == 2  # N % 8 (bf16 [K,N])
    assert L.gpt2_linear(17, 16, 16, None, 16, 10, 768, 768, 768, 0, 1, 1, 1, None) == 1  # misaligned x
    assert L.gpt2_linear(16, 16, None, None, 16, 10, 1000, 768, 1001, 1, 0, 1, 1, None) == 2  # bf16 row not 16 B
    assert L.gpt2_linear(16, 16, 16, 16, 16, 10, 1002, 768, 1004, 1, 3, 1, 0, None) == 2  # residual needs N % 4
    assert L.gpt2_attention_causal(16, 16, 2, 64, 12, 32, 1, None) == 2                  # head_dim != 64
    assert L.gpt2_attention_causal(16, 16, 0, 64, 12, 64, 1, None) == 0                  # B = 0
    assert L.gpt2_attention_causal_scaled(16, 16, 2, 64, 12, 64, 0.0, 1, None) == 1      # scale <= 0
    assert L.gpt2_attention_causal_scaled(16, 16, 2, 64, 12, 64, float("inf"), 1, None) == 1
    assert L.gpt2_attention_causal_scaled(16, 16, 0, 64, 12, 64, 0.0625, 1, None) == 0   # B = 0
    assert L.gpt2_linear(16, 16, 16, None, 16, 10, 768, 768, 768, 0, 5, 1, 1, None) == 1  # unknown epilogue
    d = G.make_dims(2, 768, 12, 3072, 50257, 1024)
    blk = G.BlockWeights(*([256] * 12))
    assert L.gpt2_block_forward(ctypes.byref(d), ctypes.byref(blk), 256, 256, 2, 64, 256, 10, None) == 3  # ws small
    assert L.gpt2_block_forward_layer(ctypes.byref(d), ctypes.byref(blk), -1, 256, 256, 2, 64, 256, 1 << 30,
                                      None) == 1  # layer < 0
    d_bad = G.make_dims(2, 768, 12, 3072, 50257, 1024, flags=4)
    assert L.gpt2_block_forward(ctypes.byref(d_bad), ctypes.byref(blk), 256, 256, 2, 64, 256, 1 << 30,
                                None) == 1  # unknown switch bit
    d_sw = G.make_dims(2, 768, 12, 2048, 50257, 1024, flags=G.SCALE_ATTN_BY_INVERSE_LAYER_IDX | G.GELU_EXACT)
    assert G.gpt2_workspace_bytes(d_sw, 8, 1024) == 2 * 8192 * 768 * 4 + 2 * 8192 * 768 * 2 + 8192 * 3 * 768 * 2 + \
        8192 * 2048 * 2  # n_inner = 2048
    grads = G.BlockGrads(*([256] * 12))
    assert L.gpt2_block_backward(ctypes.byref(d), ctypes.byref(blk), 0, 256, 512, 768, ctypes.byref(grads), 2, 64,
                                 256, 1 << 30, None) == 2  # 16-bit dims: the backward is F32 only
    d32b = G.make_dims(2, 768, 12, 3072, 50257, 1024, dtype=G.F32)
    assert G.gpt2_block_backward_workspace_bytes(d, 2, 64) == 0
    wsb = G.gpt2_block_backward_workspace_bytes(d32b, 2, 64)
    assert wsb > 0
    assert L.gpt2_block_backward(ctypes.byref(d32b), ctypes.byref(blk), 0, 256, 1 << 20, 1 << 24,
                                 ctypes.byref(grads), 2, 64, 256, wsb - 1, None) == 3  # workspace too small
    assert L.gpt2_block_backward(ctypes.byref(d32b), ctypes.byref(blk), 0, 256, 1 << 20, 256 + 4096,
                                 ctypes.byref(grads), 2, 64, 256, wsb, None) == 1  # dx_in overlaps x_in
    assert L.gpt2_block_backward(ctypes.byref(d32b), ctypes.byref(blk), 0, 256, 1 << 20, 1 << 24,
                                 ctypes.byref(grads), 1, 4097, 256, 1 << 40, None) == 2  # T > 4096
    assert L.gpt2_block_backward(ctypes.byref(d32b), ctypes.byref(blk), 0, 256, 1 << 20, 1 << 24,
                                 ctypes.byref(grads), 65536, 1, 256, 1 << 40, None) == 2  # B > 65535
    blk0 = G.BlockWeights(*([256] * 11 + [0]))
    assert L.gpt2_block_forward(ctypes.byref(d), ctypes.byref(blk0), 256, 256, 2, 64, 256, 1 << 30, None) == 1
    blocks = (G.BlockWeights * 2)(blk, blk)
    mw = G.ModelWeights(256, 256, 256, 256, ctypes.cast(blocks, ctypes.POINTER(G.BlockWeights)))
    assert L.gpt2_forward_logits(ctypes.byref(d), ctypes.byref(mw), 256, 256, 50257, 1, 2, 1025, 256, 1 << 34,
                                 None) == 1  # T > n_pos
    assert L.gpt2_forward_logits(ctypes.byref(d), ctypes.byref(mw), 256, 256, 50000, 1, 2, 64, 256, 1 << 34,
                                 None) == 1  # ld < vocab
    d32 = G.make_dims(2, 768, 12, 3072, 50257, 1024, dtype=G.F32)
    assert L.gpt2_decode_step(ctypes.byref(d32), ctypes.byref(mw), 256, 4, 64, 256, 256, 256, None, 0, 256,
                              1 << 34, None) == 2  # decode is bf16 only
    assert L.gpt2_selftest_wait_timeout(0, None) == 1  # wait limit outside 1 .. 2e9 ns
    assert L.gpt2_selftest_wait_timeout(2_000_000_001, None) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(G, "library_path", str(tmp_path / "missing.so"))
    monkeypatch.setattr(G, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        G.lib()
