"""FP64 CPU oracle for the NVFP4 W4A16 skinny decode contraction.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or call it.  It shares no
code, table or constant generator with the CUDA library in
``nvfp4_w4a16_moe_skinny_gb300/csrc``; the only module both sides use is the
seeded input generator ``nvfp4_w4a16_moe_skinny_gb300.workloads``, which holds
none of the method's arithmetic.

What each module follows (page title, section):

* ``formats``  -- NVFP4 = E2M1 weights, E4M3 scale per 16 elements along K, FP32
  per-tensor global scale: gemma-cuda-hybrid README, "Everything it has /
  Inference engine" and "Why it's NVIDIA-only ... / NVFP4-specific".
* ``gemm``     -- the M<=16 skinny product y = x . W^T: gemma-cuda-hybrid
  README, "Everything it has / Inference engine" (the tensor-core GEMM bullet).
* ``moe``      -- router top-k + softmax, expert grouping, GELU-tanh-gated
  expert FFN, weighted sum plus the always-on shared branch: TensorSharp
  docs/models/gemma4.md, sections "3.1 Per-layer (dense)", "3.2 Per-layer
  (MoE)", "4.6 MoE" and "14. Optimization opportunities / Completed
  (Expert-batched FFN)"; GELU-tanh: TensorFold issue #1048, "Steps", step 2.
* ``lm_head``  -- tied NVFP4 lm_head with greedy argmax: gemma-cuda-hybrid
  README, "Headline numbers" (bit-exact greedy) and "Everything it has".
* ``layout``   -- the repacked kernel layout written as an index function from
  its prose specification (the pages only say weights are repacked offline
  into MMA-fragment order: gemma-cuda-hybrid README, "NVFP4-specific").

Every function is parity-pinned by ``tests/test_oracle_*.py`` against closed
forms, exhaustive code tables, brute force on tiny inputs, or library routines
that the oracle does not itself call.  The pages print no worked numeric
example, so the end-to-end numbers are "parity unpinned" against the pages;
each building block is pinned to mathematics instead.
"""

from . import formats, gemm, moe, lm_head, layout  # noqa: F401
