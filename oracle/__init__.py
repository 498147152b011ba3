"""Float64 CPU oracle for the GPT-2 Pre-LN forward and the gradients of its
language-model loss (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from it.
"""
from .gpt2_ref import (  # noqa: F401
    argmax_lowest, attn_extra_scale, block_forward, causal_attention, causal_probs, conv1d, decode_step, embed,
    forward_hidden, forward_logits, forward_loss, gelu_exact, gelu_new, layer_norm, lm_head, merge_heads, mlp_forward,
    logsumexp, prefill_cache, shifted_cross_entropy, split_qkv_heads,
)
from .gpt2_grad import (  # noqa: F401
    block_backward, causal_attention_backward, conv1d_backward, gelu_exact_backward, gelu_new_backward,
    layer_norm_backward, loss_and_grads,
)
