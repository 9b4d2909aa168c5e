"""CPU oracle for the MoE layer forward with an expert-slot cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, links or executes this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
arm of ``bench.py`` use it.  It shares no code with the CUDA library; the only module both
sides use is ``workloads`` (seeded input generators, which hold none of the layer's
arithmetic).

It is a plain, slow, obviously-correct restatement in fp64 (NumPy) of what the layer computes:

* ``moe_ref``  -- router logits, top-k gating, histogram / scan / stable permutation,
  token gather, SwiGLU expert FFN (bf16 and INT4 with per-group scales), shared expert and
  gate-weighted combine, and the whole layer forward;
* ``lru_sim`` -- the expert-slot LRU cache as a list-based simulator producing the
  hit / miss / eviction / slot trace;
* ``bf16``    -- bf16 bit decoding and round-to-nearest-even, written independently of the
  generator's encoder.

Pins (closed forms, brute force, invariants) live in ``tests/test_oracle_*.py``.
The realised Zipf popularity of the synthetic routers has no closed form; it is pinned by
properties of a routed batch (tests/test_workloads.py), not by exact shares.
"""
from . import bf16, lru_sim, moe_ref  # noqa: F401
