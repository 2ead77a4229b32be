"""CPU oracle for the Any-Precision mixed-precision MoE layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call, link
or execute anything under ``oracle/``: only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.  The GPU
library shares no code with it.

Plain numpy in float64, written step by step from "PagedWeight: Efficient MoE
LLM Serving with Dynamic Quality-Aware Weight Quantization" (arXiv text):
overlaid bit-planes with per-bitwidth lookup tables (§1 and the Figure 3
caption), per-expert linear-blocks gate_up and down (§3.1), top-K routing and
routing mass (§2.1, Eq. 1), released-memory accounting (§3.1, Eq. 3) and the
fused layer: routing, the experts' gate_up with SiLU·mul, their down
projection and the weighted sum of their outputs, all in one step (§3.3).  See ``oracle/apl.py``.

Parity status per function (what pins it, see tests/test_oracle_pins.py):
  pack / unpack ............ pinned: overlay invariant, round trip, hand-derived layout points
  dequant + linear ......... pinned: identity LUT == int64 matmul, constant LUT closed form
  route_topk ............... pinned: full-sort brute force, stable argsort, mass sums to 1
  moe_layer ................ pinned: scalar-loop brute force, E=1/k=1 dense-FFN reduction
  page_bytes ............... pinned: Eq. 3 differences, closed-form sizes
  moe_layer on random LUTs . parity unpinned beyond the above (the pages print no worked example)
"""
from .apl import *  # noqa: F401,F403
