"""Plain, slow, float64 CPU oracle for exact tree-structured prefill.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` use it.  It shares no code
with the CUDA library and imports nothing from it.

What it computes (Flide, "Accelerating Decision Inference with Exact State
Forking"): every question branch of a request is run as its own ISOLATED,
unbatched pass over trunk + branch (Proposition 3.1: the forked result equals
this pass), with

* scaled dot-product causal attention (section 3.2.1, Eq. 3 visibility; the
  1/sqrt(d) scale from the attention formula of the Flex paper, "Request-
  Adaptive Execution for Efficient Hybrid LLM Inference", section 2, Eq. 1);
* the gated delta rule stepped token by token (section 3.2.2, Eq. 4);
* the option distribution over the readout row (section 3.1, Eq. 1);
* the flat-stream layout (section 3.2, Eq. 2), the visible key sets
  (Eq. 3) and copy-on-write page accounting (ForkServe README, "Copy-on-write
  context tree").

Modules: ``layout`` (stream, positions, visible sets, page counts),
``attention``, ``gdn``, ``choice``, ``numerics`` (bf16 rounding), ``forward``
(tree-level isolated passes).
"""
from . import attention, choice, forward, gdn, layout, numerics  # noqa: F401
