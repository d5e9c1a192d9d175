"""CPU oracle for the FlashAttention forward.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference arm may import, call or run anything in this
package.  The CUDA product path (attention_forward_fa_gb300) shares no code
with it and never imports it.

  attention  -- float64 definition of attention with every masking variant
  online     -- blockwise online softmax (exact fp64, or a reduced-precision
                emulation used to pin the error metrics)
  metrics    -- row gain, rel-L2, bf16 floors, order-difference noise floor

Parity status: attention.attention_fwd is pinned by closed forms, invariants,
brute force, a library softmax and the blockwise recomputation (tests marked
"not gpu"); metrics are pinned by the printed numbers of the sparse-MLA page
through the emulation in online.py.
"""
from .attention import attention_fwd, attention_problem  # noqa: F401
