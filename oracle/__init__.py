"""CPU oracle for dynamic block-sparse attention (BSA) -- TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 NumPy restatements of what the method computes, written from
the source pages and used only by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``.  The product path (the CUDA library and
its Python binding) never imports anything from here, and nothing here imports
the product path: the two share no code.  Inputs come from the seeded
generators in ``block_sparse_attention_plan_gb300.workloads``, which hold none
of the method's arithmetic.

Modules:

* ``oracle.attention`` -- masked softmax attention over the interactions a
  logical block mask selects ("Decoupling Logical Masks from GPU Execution for
  Dynamic Block-Sparse Attention" (Tessera), abstract: BSA computes only the
  blocks a logical mask selects, preserving the specified interactions).
  Two forms: a brute-force dense masked form (tiny shapes) and a per-q-block
  gather form (large shapes), checked against each other.
* ``oracle.plan`` -- the logical-mask -> physical-tile plan (Tessera abstract:
  the physical mapping layer retains, combines or subdivides logical blocks
  into physical tiles; the task organisation layer groups and schedules tiles)
  plus the GQA per-group union table ("CompactAttention", summary: Q-block
  union + intra-group union build a per-group KV block table).

Pins (what each part is checked against, other than itself) are listed in each
module's docstring.  Parity status: attention -- pinned; plan -- pinned.
"""
from . import attention, plan  # noqa: F401
