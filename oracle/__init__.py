"""Plain, slow CPU oracle for the FlexGen int4 group-quantized OPT layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only tests/, the smoke check in __graft_entry__.py and bench.py's CPU
baseline (and its --impl reference arm) may use it.  It shares no code with
the CUDA library under int4_group_quantized_gb300/.

  codec     the 4-bit group codec in IEEE fp32 (quantize, dequantize)
  layer     prefill / decode / zig-zag block in fp64
  formulas  the byte and flop counts the page prints

Every function is pinned by a CPU test under tests/ (test_oracle_*.py) to
something other than itself: the page's printed figures, hand-worked groups,
exact rational arithmetic, brute-force attention, a textbook library
attention, and the decode == last-row-of-prefill invariant.
"""
from . import codec, formulas, layer  # noqa: F401
