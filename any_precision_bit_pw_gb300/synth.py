"""Seeded synthetic inputs for the Any-Precision MoE layer workloads.

This module only draws random numbers and fixes shapes.  It holds none of the
method's arithmetic (no packing, no dequantisation, no routing, no matmul):
the GPU library and the CPU oracle both consume what it returns, and neither
depends on the other.

Shapes follow the Mixtral models named in "PagedWeight: Efficient MoE LLM
Serving with Dynamic Quality-Aware Weight Quantization" (arXiv text, §4,
Table 1: Mixtral-8x7B has 8 experts and top-2 routing); the value
distributions are these:

* parent indices are i.i.d. uniform on [0, 2^P);
* every lookup table row is 2^b fp16 centroids drawn from N(0, 0.02^2) in fp32,
  rounded to fp16 and sorted ascending (ties after rounding allowed);
* activations are N(0, 1) rounded to fp16, router logits are fp32.

Every array has its own generator, seeded from the workload seed and the
array's name, so an array can be regenerated on its own and generation order
does not matter.  Draws use ``torch.Generator`` on the requested device; a CPU
draw and a CUDA draw of the same array differ, so a test that checks GPU
output against the oracle copies the device arrays to the host.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import torch

GATE_UP = 0
DOWN = 1


@dataclass(frozen=True)
class MoEShape:
    hidden: int          # H
    intermediate: int    # I
    experts: int         # E routed experts
    top_k: int           # k
    shared: int = 0      # S shared experts (every token, weight 1): expert ids E .. E+S-1

    @property
    def total_experts(self) -> int:
        return self.experts + self.shared

    def block_shape(self, u: int) -> Tuple[int, int]:
        """(rows, cols) of a linear-block: gate_up is 2I x H, down is H x I."""
        if u == GATE_UP:
            return 2 * self.intermediate, self.hidden
        return self.hidden, self.intermediate


TINY = MoEShape(hidden=256, intermediate=512, experts=4, top_k=2)
MIXTRAL_8X7B = MoEShape(hidden=4096, intermediate=14336, experts=8, top_k=2)
MIXTRAL_8X22B = MoEShape(hidden=6144, intermediate=16384, experts=8, top_k=2)
# The pages' Table 1 gives these two models' expert counts and top-k only; the
# hidden and expert sizes below are this build's choice (Qwen1.5-MoE-like
# 2048 x 1408, and a many-small-experts 2048 x 768).
QWEN15_MOE = MoEShape(hidden=2048, intermediate=1408, experts=60, top_k=4, shared=4)
GEMMA4_LIKE = MoEShape(hidden=2048, intermediate=768, experts=128, top_k=8, shared=1)


@dataclass(frozen=True)
class Workload:
    """One synthetic MoE-layer workload.

    bits_mode:
      "uniform_choice"  q_i drawn uniformly from ``bits_choices`` per block
      "fixed"           every block at ``fixed_bits``
      "hot_cold"        experts ranked 1 and 2 by the Zipf prior at 8 bits,
                        the other blocks uniform on ``bits_choices``
    logits_mode:
      "normal"    N(0, 1)
      "uniform"   N(0,1)*0.1 + 10*[e in {2t mod E, 2t+1 mod E}]  (equal load)
      "zipf"      N(0,1) + ln(pi(e)^-s / sum_r r^-s), pi a seeded rank permutation
      "biased"    N(0,1) + a fixed per-(layer, expert) N(0,1) bias
    """
    name: str
    shape: MoEShape
    tokens: int
    parent_bits: int
    seed_bits: int
    seed: int
    bits_mode: str = "uniform_choice"
    bits_choices: Tuple[int, ...] = ()
    fixed_bits: int = 0
    logits_mode: str = "normal"
    zipf_s: float = 1.2
    layers: int = 1

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)

    @property
    def supported_bits(self) -> Tuple[int, ...]:
        return tuple(range(self.seed_bits, self.parent_bits + 1))


# The five workloads.  "seed 2/3" in the first two descriptions are APL seed
# *bitwidths*; the RNG seed of the tiny layer is 0 and the others use 1..4.
TINY_LAYER = Workload("tiny", TINY, tokens=16, parent_bits=4, seed_bits=2, seed=0,
                      bits_mode="uniform_choice", bits_choices=(2, 3, 4))
MIXTRAL_8X7B_DECODE = Workload("mixtral8x7b_decode_mixed", MIXTRAL_8X7B, tokens=32,
                               parent_bits=8, seed_bits=3, seed=1,
                               bits_mode="uniform_choice", bits_choices=(3, 4, 5, 6, 7, 8))
MIXTRAL_8X7B_SWEEP = Workload("mixtral8x7b_uniform_sweep", MIXTRAL_8X7B, tokens=64,
                              parent_bits=8, seed_bits=3, seed=2,
                              bits_mode="fixed", fixed_bits=4, logits_mode="uniform")
SWEEP_BITS = (3, 4, 5, 6, 8)
SWEEP_TOKENS = (1, 8, 64, 256)
MIXTRAL_8X22B_PREFILL = Workload("mixtral8x22b_prefill", MIXTRAL_8X22B, tokens=4096,
                                 parent_bits=8, seed_bits=3, seed=3,
                                 bits_mode="hot_cold", bits_choices=(3, 4),
                                 logits_mode="zipf")
MIXTRAL_8X7B_STACK = Workload("mixtral8x7b_stack32_decode", MIXTRAL_8X7B, tokens=128,
                              parent_bits=8, seed_bits=3, seed=4,
                              bits_mode="fixed", fixed_bits=8, logits_mode="biased",
                              layers=32)
STACK_STEPS = 64
STACK_COMMIT_EVERY = 8

QWEN15_DECODE = Workload("qwen15moe_decode_mixed", QWEN15_MOE, tokens=32, parent_bits=8, seed_bits=3, seed=5,
                         bits_mode="uniform_choice", bits_choices=(3, 4, 5, 6, 7, 8))
GEMMA4_DECODE = Workload("gemma4like_decode_mixed", GEMMA4_LIKE, tokens=32, parent_bits=8, seed_bits=3, seed=6,
                         bits_mode="uniform_choice", bits_choices=(3, 4, 5, 6, 7, 8))

WORKLOADS = {w.name: w for w in (TINY_LAYER, MIXTRAL_8X7B_DECODE, MIXTRAL_8X7B_SWEEP,
                                 MIXTRAL_8X22B_PREFILL, MIXTRAL_8X7B_STACK, QWEN15_DECODE, GEMMA4_DECODE)}


# ----------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------
def sub_seed(seed: int, *keys) -> int:
    """Deterministic 63-bit seed for one named array of one workload."""
    h = hashlib.sha256(repr((int(seed),) + tuple(keys)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(seed: int, device, *keys) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(sub_seed(seed, *keys))
    return g


def parent_indices(wl: Workload, layer: int, expert: int, u: int, device="cpu",
                   rows: Optional[int] = None, cols: Optional[int] = None) -> torch.Tensor:
    """uint8 [rows][cols] parent-bit indices, i.i.d. uniform on [0, 2^P)."""
    r, c = wl.shape.block_shape(u)
    r = rows if rows is not None else r
    c = cols if cols is not None else c
    g = _gen(wl.seed, device, "idx", layer, expert, u)
    return torch.randint(0, 1 << wl.parent_bits, (r, c), generator=g, device=device,
                         dtype=torch.uint8)


def lut(wl: Workload, layer: int, expert: int, u: int, bits: int, device="cpu",
        rows: Optional[int] = None) -> torch.Tensor:
    """fp16 [rows][2^bits]: per-row centroids, N(0, 0.02^2) drawn in fp32,
    rounded to fp16, sorted ascending."""
    r, _ = wl.shape.block_shape(u)
    r = rows if rows is not None else r
    g = _gen(wl.seed, device, "lut", layer, expert, u, bits)
    v = torch.randn((r, 1 << bits), generator=g, device=device, dtype=torch.float32) * 0.02
    return torch.sort(v.to(torch.float16), dim=-1).values.contiguous()


def zipf_ranks(wl: Workload, layer: int = 0) -> torch.Tensor:
    """pi(e): a seeded permutation of the ranks 1..E (int64, CPU)."""
    g = _gen(wl.seed, "cpu", "zipf_perm", layer)
    return torch.randperm(wl.shape.experts, generator=g) + 1


def committed_bits(wl: Workload, layer: int = 0) -> List[int]:
    """q_i for the 2(E+S) blocks of one layer (routed then shared experts),
    ordered (expert, u) with u=0 gate_up."""
    E = wl.shape.total_experts
    if wl.bits_mode == "fixed":
        return [wl.fixed_bits] * (2 * E)
    g = _gen(wl.seed, "cpu", "bits", layer)
    ch = torch.tensor(wl.bits_choices, dtype=torch.int64)
    draw = ch[torch.randint(0, len(ch), (2 * E,), generator=g)].tolist()
    if wl.bits_mode == "uniform_choice":
        return draw
    if wl.bits_mode == "hot_cold":
        ranks = zipf_ranks(wl, layer).tolist()
        return [wl.parent_bits if ranks[b // 2] <= 2 else draw[b] for b in range(2 * E)]
    raise ValueError(wl.bits_mode)


def hot_experts(wl: Workload, layer: int = 0) -> List[int]:
    """Experts whose Zipf prior rank is 1 or 2 (the hot experts of the prefill layer)."""
    ranks = zipf_ranks(wl, layer).tolist()
    return sorted(e for e in range(wl.shape.experts) if ranks[e] <= 2)


def activations(wl: Workload, layer: int = 0, step: int = 0, device="cpu",
                tokens: Optional[int] = None) -> torch.Tensor:
    """fp16 [T][H] drawn N(0, 1)."""
    T = tokens if tokens is not None else wl.tokens
    g = _gen(wl.seed, device, "x", layer, step, T)
    return torch.randn((T, wl.shape.hidden), generator=g, device=device,
                       dtype=torch.float32).to(torch.float16)


def router_logits(wl: Workload, layer: int = 0, step: int = 0, device="cpu",
                  tokens: Optional[int] = None) -> torch.Tensor:
    """fp32 [T][E] router logits for the workload's routing pattern."""
    T = tokens if tokens is not None else wl.tokens
    E = wl.shape.experts
    g = _gen(wl.seed, "cpu", "logits", layer, step, T)
    z = torch.randn((T, E), generator=g, dtype=torch.float32)
    if wl.logits_mode == "normal":
        out = z
    elif wl.logits_mode == "uniform":
        t = torch.arange(T)
        bump = torch.zeros((T, E))
        bump[t, (2 * t) % E] = 10.0
        bump[t, (2 * t + 1) % E] = 10.0
        out = z * 0.1 + bump
    elif wl.logits_mode == "zipf":
        ranks = zipf_ranks(wl, layer).to(torch.float64)
        r = torch.arange(1, E + 1, dtype=torch.float64)
        prior = torch.log(ranks ** (-wl.zipf_s) / torch.sum(r ** (-wl.zipf_s)))
        out = z + prior.to(torch.float32)
    elif wl.logits_mode == "biased":
        gb = _gen(wl.seed, "cpu", "expert_bias", layer)
        bias = torch.randn((E,), generator=gb, dtype=torch.float32)
        out = z + bias
    else:
        raise ValueError(wl.logits_mode)
    return out.to(torch.float32).contiguous().to(device)


@dataclass
class LayerInputs:
    """Everything one MoE layer call needs, as plain tensors."""
    wl: Workload
    layer: int
    bits: List[int]                                   # q_i per (expert, u)
    idx: Dict[Tuple[int, int], torch.Tensor]          # (e, u) -> uint8 [rows][cols]
    luts: Dict[Tuple[int, int], Dict[int, torch.Tensor]]  # (e, u) -> {b: fp16 [rows][2^b]}
    x: torch.Tensor                                   # fp16 [T][H]
    logits: torch.Tensor                              # fp32 [T][E]


def layer_inputs(wl: Workload, layer: int = 0, step: int = 0, device="cpu",
                 tokens: Optional[int] = None, experts: Optional[Sequence[int]] = None,
                 lut_bits: Optional[Sequence[int]] = None) -> LayerInputs:
    """Draw one layer.  ``experts`` limits which experts' weights are drawn;
    ``lut_bits`` limits which LUT bitwidths are drawn (default: all of S..P)."""
    E = wl.shape.total_experts
    ex = range(E) if experts is None else experts
    lb = wl.supported_bits if lut_bits is None else tuple(lut_bits)
    idx, luts = {}, {}
    for e in ex:
        for u in (GATE_UP, DOWN):
            idx[(e, u)] = parent_indices(wl, layer, e, u, device)
            luts[(e, u)] = {b: lut(wl, layer, e, u, b, device) for b in lb}
    return LayerInputs(wl=wl, layer=layer, bits=committed_bits(wl, layer), idx=idx, luts=luts,
                       x=activations(wl, layer, step, device, tokens),
                       logits=router_logits(wl, layer, step, device, tokens))
