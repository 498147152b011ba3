"""Seeded synthetic inputs for the GPT-2 Pre-LN forward and decode workloads.

This module is shared by the oracle-side tests, the GPU-side tests and the
benchmark. It holds only random draws, shapes and dtype rounding: none of the
model's arithmetic lives here.

Recipe (one numpy ``PCG64(seed)`` stream per workload, all draws in float64,
in this order, then rounded to the path dtype):

1. ``wte`` [V, D] and ``wpe`` [n_pos, D], both N(0, 0.02);
2. per layer: ln_1 gamma, beta; W_qkv, b_qkv; W_o, b_o; ln_2 gamma, beta;
   W_fc, b_fc; W_proj, b_proj.  Linear weights are N(0, 0.02) except the two
   output projections (attention c_proj and MLP c_proj), which are
   N(0, 0.02 / sqrt(2 * n_layer)) -- the scaled initialisation of the
   Hugging Face ``_init_weights`` described on "逐行拆GPT-2源码"
   (GPT2LMHeadModel section).  Biases are N(0, 0.01); LayerNorm gamma is
   1 + N(0, 0.02) and beta is N(0, 0.02);
3. ln_f gamma, beta;
4. then the activations X (N(0, 1)) or the token ids (uniform in [0, V));
5. then, for decode, the per-layer K/V caches (N(0, 1)).

Linear weights are stored [in, out] (the Conv1D orientation of the Hugging
Face GPT-2 code, "逐行拆GPT-2源码", GPT2Attention section), so
``y = x @ W + b``.

Values are returned as ``np.float32`` arrays whose every element is exactly
representable in the path dtype ("f32", "bf16" or "f16").  Rounding is float64 ->
float32 (round to nearest even) and, for bf16, float32 -> bf16 (round to
nearest even on the bit pattern).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Dims:
    """Model hyper-parameters, named as in the GPT2Config of the pages."""

    n_layer: int
    d_model: int
    n_head: int
    d_ff: int
    vocab: int
    n_pos: int
    eps: float = 1e-5
    # GPT2Config switches the pages name (both off for the GPT-2 workloads):
    # attention scores of layer l also divided by l + 1, and the exact GELU
    # x * Phi(x) in the MLP instead of its tanh approximation
    scale_attn_by_inverse_layer_idx: bool = False
    gelu_exact: bool = False

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_head


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    dtype: str          # "f32" or "bf16"
    B: int
    T: int
    seed: int
    kind: str           # "block" | "forward" | "decode"
    decode_steps: int = 0
    cache_len: int = 0  # prefilled cache length per sequence (decode)


GPT2_SMALL = Dims(n_layer=12, d_model=768, n_head=12, d_ff=3072, vocab=50257, n_pos=1024)
GPT2_MEDIUM = Dims(n_layer=24, d_model=1024, n_head=16, d_ff=4096, vocab=50257, n_pos=1024)
GPT2_XL = Dims(n_layer=48, d_model=1600, n_head=25, d_ff=6400, vocab=50257, n_pos=1024)
# Decode past position 1023 needs more position rows than the 1024 the pages'
# table has; the synthetic table grows to 1088 rows (1023 cached + 64 new).
GPT2_SMALL_DECODE = dataclasses.replace(GPT2_SMALL, n_pos=1088)

WORKLOADS = {
    "block_fp32_b1_t64": Workload("block_fp32_b1_t64", dataclasses.replace(GPT2_SMALL, n_layer=1),
                                  "f32", 1, 64, 1234, "block"),
    "gpt2_small_fwd_b8_t1024": Workload("gpt2_small_fwd_b8_t1024", GPT2_SMALL, "bf16", 8, 1024, 1235, "forward"),
    "gpt2_medium_fwd_b16_t1024": Workload("gpt2_medium_fwd_b16_t1024", GPT2_MEDIUM, "bf16", 16, 1024, 1236,
                                          "forward"),
    "gpt2_xl_fwd_b4_t1024": Workload("gpt2_xl_fwd_b4_t1024", GPT2_XL, "bf16", 4, 1024, 1237, "forward"),
    "gpt2_small_decode_b64": Workload("gpt2_small_decode_b64", GPT2_SMALL_DECODE, "bf16", 64, 1, 1238, "decode",
                                      decode_steps=64, cache_len=1023),
}

BLOCK_KEYS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o",
              "ln2_g", "ln2_b", "w_fc", "b_fc", "w_proj", "b_proj")


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 draws to float32 holding values exact in ``dtype``."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return x32
    if dtype == "f16":
        return x32.astype(np.float16).astype(np.float32)
    if dtype != "bf16":
        raise ValueError(f"unknown dtype {dtype!r}")
    bits = x32.view(np.uint32)
    # round to nearest even on the upper 16 bits (inputs here are finite)
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    rounded = (bits + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return rounded.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values already exact in bf16 (as uint16)."""
    x32 = np.ascontiguousarray(x, dtype=np.float32)
    return (x32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


class _Draw:
    def __init__(self, seed: int, dtype: str):
        self.rng = np.random.Generator(np.random.PCG64(seed))
        self.dtype = dtype

    def normal(self, shape, std, mean=0.0):
        z = self.rng.standard_normal(shape)
        z *= std
        if mean:
            z += mean
        return round_to(z, self.dtype)


def draw_block(d: _Draw, dims: Dims) -> dict:
    D, F = dims.d_model, dims.d_ff
    proj_std = 0.02 / math.sqrt(2 * dims.n_layer)
    blk = {}
    blk["ln1_g"] = d.normal((D,), 0.02, 1.0)
    blk["ln1_b"] = d.normal((D,), 0.02)
    blk["w_qkv"] = d.normal((D, 3 * D), 0.02)
    blk["b_qkv"] = d.normal((3 * D,), 0.01)
    blk["w_o"] = d.normal((D, D), proj_std)
    blk["b_o"] = d.normal((D,), 0.01)
    blk["ln2_g"] = d.normal((D,), 0.02, 1.0)
    blk["ln2_b"] = d.normal((D,), 0.02)
    blk["w_fc"] = d.normal((D, F), 0.02)
    blk["b_fc"] = d.normal((F,), 0.01)
    blk["w_proj"] = d.normal((F, D), proj_std)
    blk["b_proj"] = d.normal((D,), 0.01)
    return blk


def draw_model(dims: Dims, dtype: str, seed: int, with_embeddings: bool = True):
    """Return (params, draw) with params = {wte, wpe, blocks[], lnf_g, lnf_b}.

    The returned ``_Draw`` continues the same stream, so activations, tokens
    and caches drawn from it follow the recipe's order.
    """
    d = _Draw(seed, dtype)
    p = {}
    if with_embeddings:
        p["wte"] = d.normal((dims.vocab, dims.d_model), 0.02)
        p["wpe"] = d.normal((dims.n_pos, dims.d_model), 0.02)
    p["blocks"] = [draw_block(d, dims) for _ in range(dims.n_layer)]
    if with_embeddings:
        p["lnf_g"] = d.normal((dims.d_model,), 0.02, 1.0)
        p["lnf_b"] = d.normal((dims.d_model,), 0.02)
    return p, d


def draw_tokens(d: _Draw, B: int, T: int, vocab: int) -> np.ndarray:
    return d.rng.integers(0, vocab, size=(B, T), dtype=np.int64).astype(np.int32)


def draw_activations(d: _Draw, B: int, T: int, D: int) -> np.ndarray:
    """Residual-stream input X ~ N(0, 1); the residual stream is float32."""
    return round_to(d.rng.standard_normal((B, T, D)), "f32")


def kv_cache_slabs(d: _Draw, dims: Dims, B: int, T_fill: int):
    """The filled slots of the KV cache one (layer, K|V) slab at a time, in
    draw order: yields (l, kv, slab [B, H, T_fill, head_dim] ~ N(0,1), bf16
    values).  Lets a caller move a large cache to the device without holding
    it all on the host."""
    H, hd = dims.n_head, dims.head_dim
    for l in range(dims.n_layer):
        for kv in range(2):
            yield l, kv, round_to(d.rng.standard_normal((B, H, T_fill, hd)), "bf16")


def draw_kv_cache(d: _Draw, dims: Dims, B: int, T_max: int, T_fill: int) -> np.ndarray:
    """KV cache [L, 2, B, H, T_max, head_dim]; slots < T_fill ~ N(0,1) (bf16), rest 0."""
    L, H, hd = dims.n_layer, dims.n_head, dims.head_dim
    cache = np.zeros((L, 2, B, H, T_max, hd), dtype=np.float32)
    for l, kv, slab in kv_cache_slabs(d, dims, B, T_fill):
        cache[l, kv, :, :, :T_fill, :] = slab
    return cache


def param_count(params: dict) -> dict:
    """Counts per group, grouped as in the GPT-2 small parameter table."""
    att = ("w_qkv", "b_qkv", "w_o", "b_o")
    ffn = ("w_fc", "b_fc", "w_proj", "b_proj")
    ln = ("ln1_g", "ln1_b", "ln2_g", "ln2_b")
    out = {
        "wte": int(params["wte"].size),
        "wpe": int(params["wpe"].size),
        "attention": sum(int(b[k].size) for b in params["blocks"] for k in att),
        "ffn": sum(int(b[k].size) for b in params["blocks"] for k in ffn),
        "layernorm": sum(int(b[k].size) for b in params["blocks"] for k in ln)
        + int(params["lnf_g"].size) + int(params["lnf_b"].size),
    }
    out["total"] = sum(out.values())
    return out


def param_shapes(dims: Dims) -> dict:
    """Shapes of every tensor, without drawing (for counting large models)."""
    D, F = dims.d_model, dims.d_ff
    blk = {"ln1_g": (D,), "ln1_b": (D,), "w_qkv": (D, 3 * D), "b_qkv": (3 * D,), "w_o": (D, D), "b_o": (D,),
           "ln2_g": (D,), "ln2_b": (D,), "w_fc": (D, F), "b_fc": (F,), "w_proj": (F, D), "b_proj": (D,)}
    return {"wte": (dims.vocab, D), "wpe": (dims.n_pos, D), "block": blk, "lnf_g": (D,), "lnf_b": (D,)}


def workload_inputs(name: str, T_override: int | None = None, B_override: int | None = None,
                    cache_as_slabs: bool = False):
    """Draw every input of a named workload, in recipe order.

    Returns a dict with ``dims``, ``dtype``, ``params`` and either ``x``
    (block workloads) or ``tokens`` (forward / decode workloads); decode
    workloads also get ``cache`` (filled slots ``cache_len``) and
    ``past_len``; with ``cache_as_slabs`` the cache comes as the generator
    of ``kv_cache_slabs`` (``cache_slabs``) instead, to be consumed after
    everything else has been drawn.
    """
    w = WORKLOADS[name]
    B = B_override or w.B
    T = T_override or w.T
    out = {"workload": w, "dims": w.dims, "dtype": w.dtype, "B": B, "T": T}
    if w.kind == "block":
        params, d = draw_model(w.dims, w.dtype, w.seed, with_embeddings=False)
        out["params"] = params
        out["x"] = draw_activations(d, B, T, w.dims.d_model)
    elif w.kind == "forward":
        params, d = draw_model(w.dims, w.dtype, w.seed)
        out["params"] = params
        out["tokens"] = draw_tokens(d, B, T, w.dims.vocab)
    else:
        params, d = draw_model(w.dims, w.dtype, w.seed)
        out["params"] = params
        out["tokens"] = draw_tokens(d, B, 1, w.dims.vocab)[:, 0]
        T_max = w.cache_len + w.decode_steps
        out["T_max"] = T_max
        if cache_as_slabs:
            out["cache_slabs"] = kv_cache_slabs(d, w.dims, B, w.cache_len)
        else:
            out["cache"] = draw_kv_cache(d, w.dims, B, T_max, w.cache_len)
        out["past_len"] = np.full((B,), w.cache_len, dtype=np.int32)
    return out


def convert_params(params: dict, dtype: str) -> dict:
    """The same parameters rounded to another path dtype (e.g. a bf16 model's
    weights as fp16 operands: exact for magnitudes from 2^-17 up)."""
    out = {k: round_to(v, dtype) for k, v in params.items() if k != "blocks"}
    out["blocks"] = [{k: round_to(v, dtype) for k, v in b.items()} for b in params["blocks"]]
    return out


def replace_dims(d: Dims, **kw) -> Dims:
    """A copy of ``d`` with some fields changed (e.g. fewer layers)."""
    return dataclasses.replace(d, **kw)
