"""Plain fp64 CPU oracle for paged decode attention, LSE merge and ragged causal prefill.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the C-ABI library and its Python binding) never
calls it, and this package imports nothing from the product package: the two
share no code.  Seeded inputs come from ``paged_kv_attention_32_gb300.workloads``,
which holds no attention arithmetic.

Every function follows a definition printed on the FlashInfer API pages
``batch_decode_with_paged_kv_cache`` (prims_ts), ``cudnn_batch_decode_with_kv_cache``
and ``batch_prefill`` (prims_ts); the docstrings cite the page and parameter.
bf16 and fp16 inputs are taken as raw uint16 bit patterns and widened to
float64 exactly (from each format's definition), so the oracle needs no
16-bit float support from any library.
"""

from .attention import (  # noqa: F401
    LOG2E,
    bf16_bits_to_f64,
    f16_bits_to_f64,
    bits_to_f64,
    gather_kv,
    decode_row_key_range,
    attention_rows,
    paged_decode_request,
    paged_decode,
    merge_states,
    prefill_request,
    batch_prefill,
)
from .plan_spec import plan_spec  # noqa: F401
