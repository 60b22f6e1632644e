"""CPU oracle for the W4A16 linear layer C = A . dequant(W) (+ bias).

TEST INFRASTRUCTURE ONLY. Nothing in the library imports, links or calls this
package; only tests/, the smoke check in __graft_entry__.py and the CPU
baseline leg of bench.py use it. It shares no code with the CUDA path: the two
meet only on the seeded inputs from the separate ``synth`` module.

Modules:
  ieee   binary16 / bfloat16 decoding and round-to-nearest-even encoding (fp64)
  w4a16  pack / unpack / dequant / fp64 product / tolerance predicate
  exact  rational-arithmetic brute force for tiny problems (independent decoder)

Every function is pinned by tests in tests/test_oracle_pins.py against values
the pages print, closed forms, invariants, library conversions and brute force.
Parity unpinned: none of the functions; the pages print no numeric input/output
values for the product, so its pins are closed forms, invariants and brute
force rather than published numbers.
"""
from . import ieee, w4a16, exact  # noqa: F401
from .w4a16 import *  # noqa: F401,F403
