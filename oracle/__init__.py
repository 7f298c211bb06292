"""CPU oracle for one block-diffusion drafter cycle (DFlash drafter + DDTree).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this package: only the test-suite, the smoke check and the CPU
baseline leg of the benchmark do.  The CUDA library shares no code, header,
table or helper with it; the two meet only in the seeded input generator.

The oracle restates what the pages define, step by step, in NumPy float64
(float32 where the pages' algorithm fixes a float32 decision, namely the tree
scores), with no tiling, fusion or reordering:

* ``drafter``  - feature fusion, KV injection, the drafter block pass,
                 log-softmax and top-K ("DFlash: Block Diffusion for Flash
                 Speculative Decoding", sections 3.4.3-3.4.4; "Accelerating
                 Speculative Decoding with Block Diffusion Draft Trees",
                 section 3.4.2);
* ``ddtree``   - Algorithm 1 (best-first heap over rank tuples), the tree
                 attention mask and the verifier walk (DDTree page, sections
                 3.4.3-3.4.5);
* ``cycle``    - the speedup identity of Equation 1 (DFlash page, 3.4.1).

Each function is pinned by tests in ``tests/test_oracle_*.py`` against facts
the pages or mathematics fix (worked examples, closed forms, brute force,
independent formulations).
"""
from . import cycle, ddtree, drafter  # noqa: F401
