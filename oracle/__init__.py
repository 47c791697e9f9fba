"""CPU oracle for the block-scaled FP4 MoE FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA library and never consumes a value the CUDA
library produced, except where a test deliberately feeds it the GPU's routing
(``forced_ids``) to compare downstream stages on identical decisions.

It is a plain, slow, obviously-correct restatement of what the layer
computes, in float64 with explicit rounding to float32 / BF16 at the stage
boundaries where a result is materialised in that precision:

* ``formats``  -- E2M1, E8M0, E4M3 and BF16 decoding, OCP MXFP4 block
                  quantisation, NVFP4 dequantisation and NVFP4 -> MXFP4
                  re-quantisation.
* ``moe``      -- router logits, softmax, top-k, renormalisation, the
                  token-to-expert permutation, routed SwiGLU experts on MXFP4
                  activations, the BF16 shared expert and the weighted combine.

Every function is pinned by ``tests/test_oracle_*.py`` against facts fixed
outside the oracle (exhaustive library decodes, closed forms, brute force,
invariants).  No function here is "parity unpinned".
"""
from . import formats, moe  # noqa: F401
