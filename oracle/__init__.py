"""CPU oracle for paged-KV decode attention and KV append.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the ``libpkv`` C-ABI
library or its Python binding) imports, calls or links anything in this
package. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may use it.

The oracle is plain and slow on purpose:

* ``paged_attention`` -- float64 single-query attention that walks each
  sequence's block table token by token (logical position -> physical block,
  row) and evaluates ``softmax(scale * q K^T) V`` with a max-subtracted
  softmax. It also holds the partial-state merge (the split-K identity) and
  the multi-query (speculative verification / prefill chunk) causal variant.
* ``append`` -- the KV-cache write: a bit copy for fp16/bf16 caches and the
  INT8 quantise-on-append rule with per-(block, kv_head) fp32 scales, written
  with NumPy float32 operations so that each IEEE round-to-nearest step is the
  same one the kernel takes. Also the copy-on-write block copy.

Conventions: ``np.uint16`` arrays hold bfloat16 bit patterns, ``np.float16``
arrays hold fp16 values, ``np.int8`` arrays hold quantised codes. Caches are
laid out ``[num_blocks, num_kv_heads, block_size, head_dim]``.

Sources: the four pages describe a paged KV cache as a pool of fixed-size
physical blocks reached through a per-sequence logical->physical page table,
gathered inside the attention kernel with no compaction copy
(Continuous-Batching-LLM-Inference-Engine README, feature list "Paged
KV-cache" and "PagedAttention kernel"), paged INT8 KV storage
(paged-inference-engine overview), and a paged KV cache that the Llama forward
"writes and reads" (mini-inference-engine, Connections). The pages print no
formula, layout or worked example; where they are silent the oracle takes the
readings documented in each function.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, brute force and hand-worked fixtures under
``tests/golden/``; none is "parity unpinned".
"""

from .paged_attention import (  # noqa: F401
    decode_kv,
    paged_decode_attention,
    paged_multiquery_attention,
    partial_state,
    merge_states,
)
from .append import (  # noqa: F401
    append_copy,
    append_int8,
    quantize_int8,
    requantize_int8,
    bf16_bits_to_f32,
    copy_blocks,
)
