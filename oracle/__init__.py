"""Plain fp64 CPU oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg (``cpu_baseline`` / ``--impl reference``) use it. It
shares no code, header, table or helper with the CUDA path.

Every function materialises the score matrix S and the probabilities P
for one (batch, head) at a time and follows the definitions on the page
"FlashAttention：快速且内存高效的准确注意力机制" (cloud.tencent.com.cn);
section names below refer to that page.

Parity status: every function here is pinned by tests under
``tests/test_oracle_*.py`` (worked mask examples, closed forms,
invariants, an independent library routine and finite differences).
The dropout generator ``philox4x32_10`` is pinned by the published
known-answer vectors of Philox4x32-10 (Random123's kat_vectors), besides
independently inverted rounds and output statistics.
"""
from .attention import (  # noqa: F401
    live_mask,
    alibi_bias,
    head_fwd,
    head_bwd,
    head_partial,
    combine_partials,
    attention_fwd,
    attention_bwd,
    decode_splitkv,
    kv_head,
    attention_fwd_varlen,
    attention_bwd_varlen,
    decode_paged,
    rotary,
    round_bf16,
    decode_kvcache,
    philox4x32_10,
    dropout_threshold,
    dropout_scale_matrix,
    attention_fwd_dropout,
    attention_bwd_dropout,
)
