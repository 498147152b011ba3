"""Python binding of libgpt2gb, the GB300 (sm_103a) GPT-2 Pre-LN forward library.

Thin ctypes marshalling over the C ABI of ``include/gpt2gb.h``: every
function here has the name of the C entry point it calls, takes device
tensors (or raw integer pointers) and sizes, and raises ``GPT2Error`` on a
non-zero status.  All arithmetic runs in the CUDA library; if the library is
missing the calls raise instead of falling back to anything else.
PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "GPT2Error", "F32", "BF16", "F16", "EPI_NONE", "EPI_BIAS", "EPI_BIAS_GELU", "EPI_BIAS_RESIDUAL",
    "EPI_BIAS_GELU_EXACT", "SCALE_ATTN_BY_INVERSE_LAYER_IDX", "GELU_EXACT", "W_IN_OUT", "W_OUT_IN", "Dims", "BlockWeights", "ModelWeights", "lib", "library_path", "gpt2_abi_version",
    "gpt2_status_string", "gpt2_last_error", "gpt2_selftest_wait_timeout", "gpt2_layernorm", "gpt2_linear", "gpt2_attention_causal",
    "gpt2_attention_causal_scaled", "gpt2_attention_causal_lse", "gpt2_attention_backward_workspace_bytes",
    "gpt2_attention_causal_backward", "gpt2_block_forward_layer", "BlockGrads", "block_grads",
    "gpt2_block_backward_workspace_bytes", "gpt2_block_backward", "ModelGrads", "model_grads",
    "gpt2_train_workspace_bytes", "gpt2_forward_backward",
    "gpt2_mlp_workspace_bytes", "gpt2_mlp", "gpt2_mlp_noalloc", "gpt2_mlp_noalloc_max_scratch_bytes",
    "gpt2_workspace_bytes", "gpt2_block_forward", "gpt2_forward_logits", "gpt2_loss_workspace_bytes",
    "gpt2_forward_loss", "gpt2_prefill_workspace_bytes", "gpt2_prefill",
    "gpt2_kv_cache_bytes", "gpt2_decode_workspace_bytes", "gpt2_decode_step", "gpt2_profile_begin",
    "gpt2_profile_end", "gpt2_profile_read", "ProfileEntry",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
# the in-tree build, or another build of the same sources named by GPT2GB_LIBRARY
library_path = os.environ.get("GPT2GB_LIBRARY") or os.path.join(_PKG, "libgpt2gb.so")

F32, BF16, F16 = 0, 1, 2
EPI_NONE, EPI_BIAS, EPI_BIAS_GELU, EPI_BIAS_RESIDUAL, EPI_BIAS_GELU_EXACT = 0, 1, 2, 3, 4
# GPT2Config switches (gpt2_dims.flags)
SCALE_ATTN_BY_INVERSE_LAYER_IDX, GELU_EXACT = 1, 2
W_IN_OUT, W_OUT_IN = 0, 1

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape or type", 3: "workspace too small",
           4: "CUDA error", 5: "device wait timed out", 6: "token id or position out of range"}


class GPT2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({_STATUS.get(status, 'unknown')})")


class Dims(ctypes.Structure):
    _fields_ = [("n_layer", ctypes.c_int), ("d_model", ctypes.c_int), ("n_head", ctypes.c_int),
                ("d_ff", ctypes.c_int), ("vocab", ctypes.c_int), ("n_pos", ctypes.c_int), ("eps", ctypes.c_float),
                ("dtype", ctypes.c_int), ("flags", ctypes.c_uint)]


_BLOCK_FIELDS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_o", "b_o", "ln2_g", "ln2_b", "w_fc", "b_fc", "w_proj",
                 "b_proj")


class BlockWeights(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in _BLOCK_FIELDS]


class BlockGrads(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in _BLOCK_FIELDS]


class ModelGrads(ctypes.Structure):
    _fields_ = [("wte", ctypes.c_void_p), ("wpe", ctypes.c_void_p), ("lnf_g", ctypes.c_void_p),
                ("lnf_b", ctypes.c_void_p), ("blocks", ctypes.POINTER(BlockGrads))]


class ModelWeights(ctypes.Structure):
    _fields_ = [("wte", ctypes.c_void_p), ("wpe", ctypes.c_void_p), ("lnf_g", ctypes.c_void_p),
                ("lnf_b", ctypes.c_void_p), ("blocks", ctypes.POINTER(BlockWeights))]


class ProfileEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int), ("ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


_lib = None
_VP, _I64, _I32, _SZ, _F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_SIGS = {
    "gpt2_abi_version": (_I32, []),
    "gpt2_status_string": (ctypes.c_char_p, [_I32]),
    "gpt2_last_error": (_I32, [ctypes.POINTER(ctypes.c_int)]),
    "gpt2_selftest_wait_timeout": (_I32, [ctypes.c_uint64, _VP]),
    "gpt2_layernorm": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _F, _I32, _I32, _VP]),
    "gpt2_linear": (_I32, [_VP, _VP, _VP, _VP, _VP, _I64, _I32, _I32, _I64, _I32, _I32, _I32, _I32, _VP]),
    "gpt2_attention_causal": (_I32, [_VP, _VP, _I32, _I32, _I32, _I32, _I32, _VP]),
    "gpt2_attention_causal_scaled": (_I32, [_VP, _VP, _I32, _I32, _I32, _I32, _F, _I32, _VP]),
    "gpt2_attention_causal_lse": (_I32, [_VP, _VP, _VP, _I32, _I32, _I32, _I32, _F, _I32, _VP]),
    "gpt2_attention_backward_workspace_bytes": (_SZ, [_I32, _I32, _I32]),
    "gpt2_attention_causal_backward": (_I32, [_VP, _VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32, _F, _VP, _SZ, _I32,
                                              _VP]),
    "gpt2_mlp_workspace_bytes": (_SZ, [_I64, _I32, _I32]),
    "gpt2_mlp": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I32, _I32, _VP, _SZ, _I32, _VP]),
    "gpt2_workspace_bytes": (_SZ, [ctypes.POINTER(Dims), _I32, _I32]),
    "gpt2_block_forward": (_I32, [ctypes.POINTER(Dims), ctypes.POINTER(BlockWeights), _VP, _VP, _I32, _I32, _VP, _SZ,
                                  _VP]),
    "gpt2_block_forward_layer": (_I32, [ctypes.POINTER(Dims), ctypes.POINTER(BlockWeights), _I32, _VP, _VP, _I32, _I32,
                                        _VP, _SZ, _VP]),
    "gpt2_block_backward_workspace_bytes": (_SZ, [ctypes.POINTER(Dims), _I32, _I32]),
    "gpt2_block_backward": (_I32, [ctypes.POINTER(Dims), ctypes.POINTER(BlockWeights), _I32, _VP, _VP, _VP,
                                   ctypes.POINTER(BlockGrads), _I32, _I32, _VP, _SZ, _VP]),
    "gpt2_forward_logits": (_I32, [ctypes.POINTER(Dims), ctypes.POINTER(ModelWeights), _VP, _VP, _I64, _I32, _I32,
                                   _I32, _VP, _SZ, _VP]),
    "gpt2_loss_workspace_bytes": (_SZ, [ctypes.POINTER(Dims), _I32, _I32]),
    "gpt2_forward_loss": (_I32, [ctypes.POINTER(Dims), ctypes.POINTER(ModelWeights), _VP, _VP, _VP, _VP, _VP, _I32,
                                 _I32, _VP, _SZ, _VP]),
    "gpt2_train_workspace_bytes": (_SZ, [ctypes.POINTER(Dims), _I32, _I32]),
    "gpt2_forward_backward": (_I32, [ctypes.POINTER(Dims), ctypes.POINTER(ModelWeights), _VP, _VP,
                                     ctypes.POINTER(ModelGrads), _VP, _I32, _I32, _VP, _SZ, _VP]),
    "gpt2_kv_cache_bytes": (_SZ, [ctypes.POINTER(Dims), _I32, _I32]),
    "gpt2_decode_workspace_bytes": (_SZ, [ctypes.POINTER(Dims), _I32]),
    "gpt2_prefill_workspace_bytes": (_SZ, [ctypes.POINTER(Dims), _I32, _I32]),
    "gpt2_prefill": (_I32, [ctypes.POINTER(Dims), ctypes.POINTER(ModelWeights), _VP, _I32, _I32, _VP, _I32, _VP, _VP,
                            _VP, _I64, _VP, _SZ, _VP]),
    "gpt2_decode_step": (_I32, [ctypes.POINTER(Dims), ctypes.POINTER(ModelWeights), _VP, _I32, _I32, _VP, _VP, _VP,
                                _VP, _I64, _VP, _SZ, _VP]),
    "gpt2_mlp_noalloc_max_scratch_bytes": (_SZ, []),
    "gpt2_mlp_noalloc": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I32, _I32, _I32, _VP]),
    "gpt2_profile_begin": (_I32, [_I32]),
    "gpt2_profile_end": (_I32, []),
    "gpt2_profile_read": (_I32, [ctypes.POINTER(ProfileEntry), _I32, ctypes.POINTER(ctypes.c_int)]),
}


def lib():
    """Load libgpt2gb.so (built by ``gpt_pre_ln_gb300.build``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is missing: run `python -m gpt_pre_ln_gb300.build` first")
        L = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != 0:
        raise GPT2Error(status, where)


# ------------------------------------------------------------- entry points
def gpt2_abi_version() -> int:
    return lib().gpt2_abi_version()


def gpt2_status_string(status: int) -> str:
    return lib().gpt2_status_string(status).decode()


def gpt2_last_error():
    """(status, site) of the first device-side fault since the last call."""
    site = ctypes.c_int(0)
    st = lib().gpt2_last_error(ctypes.byref(site))
    return st, site.value


def gpt2_selftest_wait_timeout(limit_ns, stream=None):
    _check(lib().gpt2_selftest_wait_timeout(int(limit_ns), _stream(stream)), "gpt2_selftest_wait_timeout")


def gpt2_layernorm(x, gamma, beta, y, rows, D, eps, x_t, y_t, stream=None):
    _check(lib().gpt2_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(y), rows, D, eps, x_t, y_t, _stream(stream)),
           "gpt2_layernorm")


def gpt2_linear(x, w, bias, residual, y, M, N, K, ldy, w_layout, epilogue, dtype, y_t, stream=None):
    _check(lib().gpt2_linear(_ptr(x), _ptr(w), _ptr(bias), _ptr(residual), _ptr(y), M, N, K, ldy, w_layout, epilogue,
                             dtype, y_t, _stream(stream)), "gpt2_linear")


def gpt2_attention_causal(qkv, out, B, T, n_head, head_dim, dtype, stream=None):
    _check(lib().gpt2_attention_causal(_ptr(qkv), _ptr(out), B, T, n_head, head_dim, dtype, _stream(stream)),
           "gpt2_attention_causal")


def gpt2_attention_causal_scaled(qkv, out, B, T, n_head, head_dim, score_scale, dtype, stream=None):
    _check(lib().gpt2_attention_causal_scaled(_ptr(qkv), _ptr(out), B, T, n_head, head_dim, score_scale, dtype,
                                              _stream(stream)), "gpt2_attention_causal_scaled")


def gpt2_attention_causal_lse(qkv, out, lse, B, T, n_head, head_dim, score_scale, dtype, stream=None):
    _check(lib().gpt2_attention_causal_lse(_ptr(qkv), _ptr(out), _ptr(lse), B, T, n_head, head_dim, score_scale,
                                           dtype, _stream(stream)), "gpt2_attention_causal_lse")


def gpt2_attention_backward_workspace_bytes(B, T, n_head) -> int:
    return lib().gpt2_attention_backward_workspace_bytes(B, T, n_head)


def gpt2_attention_causal_backward(qkv, out, lse, dout, dqkv, B, T, n_head, head_dim, score_scale, ws, ws_bytes,
                                   dtype, stream=None):
    _check(lib().gpt2_attention_causal_backward(_ptr(qkv), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dqkv), B, T,
                                                n_head, head_dim, score_scale, _ptr(ws), ws_bytes, dtype,
                                                _stream(stream)), "gpt2_attention_causal_backward")


def gpt2_mlp_workspace_bytes(M, F, dtype) -> int:
    return lib().gpt2_mlp_workspace_bytes(M, F, dtype)


def gpt2_mlp(x, w_fc, b_fc, w_proj, b_proj, residual, out, M, D, F, ws, ws_bytes, dtype, stream=None):
    _check(lib().gpt2_mlp(_ptr(x), _ptr(w_fc), _ptr(b_fc), _ptr(w_proj), _ptr(b_proj), _ptr(residual), _ptr(out), M,
                          D, F, _ptr(ws), ws_bytes, dtype, _stream(stream)), "gpt2_mlp")


def gpt2_mlp_noalloc_max_scratch_bytes() -> int:
    return lib().gpt2_mlp_noalloc_max_scratch_bytes()


def gpt2_mlp_noalloc(x, w_fc, b_fc, w_proj, b_proj, residual, out, M, D, F, dtype, stream=None):
    """gpt2_mlp with the library's own fixed scratch instead of a workspace."""
    _check(lib().gpt2_mlp_noalloc(_ptr(x), _ptr(w_fc), _ptr(b_fc), _ptr(w_proj), _ptr(b_proj), _ptr(residual),
                                  _ptr(out), M, D, F, dtype, _stream(stream)), "gpt2_mlp_noalloc")


def gpt2_workspace_bytes(dims: Dims, B: int, T: int) -> int:
    return lib().gpt2_workspace_bytes(ctypes.byref(dims), B, T)


def gpt2_block_forward(dims: Dims, w: BlockWeights, x_in, x_out, B, T, ws, ws_bytes, stream=None):
    _check(lib().gpt2_block_forward(ctypes.byref(dims), ctypes.byref(w), _ptr(x_in), _ptr(x_out), B, T, _ptr(ws),
                                    ws_bytes, _stream(stream)), "gpt2_block_forward")


def gpt2_block_forward_layer(dims: Dims, w: BlockWeights, layer, x_in, x_out, B, T, ws, ws_bytes, stream=None):
    _check(lib().gpt2_block_forward_layer(ctypes.byref(dims), ctypes.byref(w), layer, _ptr(x_in), _ptr(x_out), B, T,
                                          _ptr(ws), ws_bytes, _stream(stream)), "gpt2_block_forward_layer")


def gpt2_block_backward_workspace_bytes(dims: Dims, B: int, T: int) -> int:
    return lib().gpt2_block_backward_workspace_bytes(ctypes.byref(dims), B, T)


def gpt2_block_backward(dims: Dims, w: BlockWeights, layer, x_in, dx_out, dx_in, grads: BlockGrads, B, T, ws,
                        ws_bytes, stream=None):
    _check(lib().gpt2_block_backward(ctypes.byref(dims), ctypes.byref(w), layer, _ptr(x_in), _ptr(dx_out),
                                     _ptr(dx_in), ctypes.byref(grads), B, T, _ptr(ws), ws_bytes, _stream(stream)),
           "gpt2_block_backward")


def gpt2_forward_logits(dims: Dims, w: ModelWeights, tokens, logits, ld, logits_t, B, T, ws, ws_bytes, stream=None):
    _check(lib().gpt2_forward_logits(ctypes.byref(dims), ctypes.byref(w), _ptr(tokens), _ptr(logits), ld, logits_t,
                                     B, T, _ptr(ws), ws_bytes, _stream(stream)), "gpt2_forward_logits")


def gpt2_loss_workspace_bytes(dims: Dims, B: int, T: int) -> int:
    return lib().gpt2_loss_workspace_bytes(ctypes.byref(dims), B, T)


def gpt2_forward_loss(dims: Dims, w: ModelWeights, tokens, labels, token_loss, lse, mean_loss, B, T, ws, ws_bytes,
                      stream=None):
    _check(lib().gpt2_forward_loss(ctypes.byref(dims), ctypes.byref(w), _ptr(tokens), _ptr(labels), _ptr(token_loss),
                                   _ptr(lse), _ptr(mean_loss), B, T, _ptr(ws), ws_bytes, _stream(stream)),
           "gpt2_forward_loss")


def gpt2_train_workspace_bytes(dims: Dims, B: int, T: int) -> int:
    return lib().gpt2_train_workspace_bytes(ctypes.byref(dims), B, T)


def gpt2_forward_backward(dims: Dims, w: ModelWeights, tokens, labels, grads: ModelGrads, mean_loss, B, T, ws,
                          ws_bytes, stream=None):
    _check(lib().gpt2_forward_backward(ctypes.byref(dims), ctypes.byref(w), _ptr(tokens), _ptr(labels),
                                       ctypes.byref(grads), _ptr(mean_loss), B, T, _ptr(ws), ws_bytes,
                                       _stream(stream)), "gpt2_forward_backward")


def gpt2_kv_cache_bytes(dims: Dims, B: int, T_max: int) -> int:
    return lib().gpt2_kv_cache_bytes(ctypes.byref(dims), B, T_max)


def gpt2_decode_workspace_bytes(dims: Dims, B: int) -> int:
    return lib().gpt2_decode_workspace_bytes(ctypes.byref(dims), B)


def gpt2_prefill_workspace_bytes(dims: Dims, B: int, T: int) -> int:
    return lib().gpt2_prefill_workspace_bytes(ctypes.byref(dims), B, T)


def gpt2_prefill(dims: Dims, w: ModelWeights, tokens, B, T, kv_cache, T_max, past_len, next_tokens, logits_opt, ld,
                 ws, ws_bytes, stream=None):
    _check(lib().gpt2_prefill(ctypes.byref(dims), ctypes.byref(w), _ptr(tokens), B, T, _ptr(kv_cache), T_max,
                              _ptr(past_len), _ptr(next_tokens), _ptr(logits_opt), ld, _ptr(ws), ws_bytes,
                              _stream(stream)), "gpt2_prefill")


def gpt2_decode_step(dims: Dims, w: ModelWeights, kv_cache, B, T_max, past_len, tokens, next_tokens, logits_opt, ld,
                     ws, ws_bytes, stream=None):
    _check(lib().gpt2_decode_step(ctypes.byref(dims), ctypes.byref(w), _ptr(kv_cache), B, T_max, _ptr(past_len),
                                  _ptr(tokens), _ptr(next_tokens), _ptr(logits_opt), ld, _ptr(ws), ws_bytes,
                                  _stream(stream)), "gpt2_decode_step")


def gpt2_profile_begin(max_launches: int):
    _check(lib().gpt2_profile_begin(max_launches), "gpt2_profile_begin")


def gpt2_profile_end():
    _check(lib().gpt2_profile_end(), "gpt2_profile_end")


def gpt2_profile_read(max_entries: int = 64):
    """{kernel name: (launches, ms, flops, bytes)} of the last profiled span."""
    arr = (ProfileEntry * max_entries)()
    n = ctypes.c_int(0)
    _check(lib().gpt2_profile_read(arr, max_entries, ctypes.byref(n)), "gpt2_profile_read")
    return {arr[i].name.decode(): (arr[i].launches, arr[i].ms, arr[i].flops, arr[i].bytes)
            for i in range(min(n.value, max_entries))}


# ------------------------------------------------------ weight marshalling
def make_dims(n_layer, d_model, n_head, d_ff, vocab, n_pos, eps=1e-5, dtype=BF16, flags=0) -> Dims:
    return Dims(n_layer, d_model, n_head, d_ff, vocab, n_pos, eps, dtype, flags)


def block_weights(tensors: dict) -> BlockWeights:
    """BlockWeights from a dict of device tensors keyed like the C struct."""
    return BlockWeights(*[_ptr(tensors[k]) for k in _BLOCK_FIELDS])


def block_grads(tensors: dict) -> BlockGrads:
    """BlockGrads from a dict of fp32 device tensors keyed like the C struct."""
    return BlockGrads(*[_ptr(tensors[k]) for k in _BLOCK_FIELDS])


def model_weights(tensors: dict):
    """(ModelWeights, keep-alive) from {wte, wpe, lnf_g, lnf_b, blocks: [dict]}."""
    blocks = (BlockWeights * len(tensors["blocks"]))(*[block_weights(b) for b in tensors["blocks"]])
    mw = ModelWeights(_ptr(tensors["wte"]), _ptr(tensors["wpe"]), _ptr(tensors["lnf_g"]), _ptr(tensors["lnf_b"]),
                      ctypes.cast(blocks, ctypes.POINTER(BlockWeights)))
    return mw, blocks


def model_grads(tensors: dict):
    """(ModelGrads, keep-alive) from {wte, wpe, lnf_g, lnf_b, blocks: [dict]} of fp32 device tensors."""
    blocks = (BlockGrads * len(tensors["blocks"]))(*[block_grads(b) for b in tensors["blocks"]])
    mg = ModelGrads(_ptr(tensors["wte"]), _ptr(tensors["wpe"]), _ptr(tensors["lnf_g"]), _ptr(tensors["lnf_b"]),
                    ctypes.cast(blocks, ctypes.POINTER(BlockGrads)))
    return mg, blocks


def to_device(params: dict, dtype: int, device="cuda"):
    """Copy a parameter dict of float32 numpy arrays to device tensors.

    Arrays are converted to bf16 (``dtype == BF16``), fp16 (``F16``) or kept
    fp32; the values are expected to be exactly representable already.  Returns the same
    nesting ({..., "blocks": [dict]}) with torch tensors.
    """
    import numpy as np
    import torch
    tdt = {BF16: torch.bfloat16, F16: torch.float16}.get(dtype, torch.float32)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device=device).to(tdt).contiguous()

    out = {k: up(v) for k, v in params.items() if k != "blocks"}
    out["blocks"] = [{k: up(v) for k, v in b.items()} for b in params["blocks"]]
    return out
