"""CPU oracle for packed prefix-tree attention, tree RoPE and letter readout.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
anything in this package: only the test suite, the package's smoke check and
the benchmark's CPU-baseline leg (and its ``--impl reference`` arm) use it.

The oracle is a plain, slow, float64 restatement of what the basal-rs
Architecture page says the path computes:

* ``plan``     -- the packing of a batch's prompts into prefix trees and one
                  token row ("03 / Packing: Attention over tree blocks",
                  "01 / Request path: Batch and prefix tree");
* ``rope``     -- rotary positions taken as the token's position in its own
                  prompt ("03 / Packing: Attention over tree blocks");
* ``attention``-- attention over tree blocks, written as its plain definition:
                  every root-to-leaf prompt is materialised as its own sequence
                  and run through dense causal attention, because the page states
                  that the tree result matches computing each full prompt
                  separately ("03 / Packing", the Q1 order-2 example);
* ``readout``  -- the two-order average and temperature calibration
                  ("02 / Basal protocol: Two option orders and calibration").

It shares no code with the CUDA library; the only common module is ``synth``,
which draws the seeded inputs and holds none of the method's arithmetic.

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against values printed on the page, closed forms, library routines on special
cases, and brute force on tiny inputs.  No function is left unpinned.
"""
from . import plan, rope, attention, readout  # noqa: F401
