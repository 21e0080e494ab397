"""CPU oracle for the single-GPU MoE layer forward (float64, numpy).

TEST INFRASTRUCTURE ONLY.  This package states what the layer computes, in
the plainest form, so that the CUDA path can be checked against it.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the library in ``moe_expert_ffn_sqrt_gb300``
never does, and the two share no code.

Every function is pinned by a ``-m "not gpu"`` test against something other
than itself (printed worked examples, closed forms, library decoders,
brute force); see ``tests/test_oracle_*.py``.
"""
from . import formats, moe  # noqa: F401
