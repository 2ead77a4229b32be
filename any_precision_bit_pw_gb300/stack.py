"""The 32-layer decode stack workload: a seeded commit schedule over the page
table, run at step boundaries.

"PagedWeight" arXiv text: the weight page table records the committed
bitwidth q_i of every per-expert linear-block (§3, §3.1); lowering a block
releases M_i^b - M_i^b' bytes (Eq. 3); routing mass (Eq. 1) measures how much
traffic an expert receives, and hot experts are protected (§3.2); commits
happen only at safe boundaries (§3.3).  The paper's planner (Algorithm 1,
Eqs. 4-8) is not built here.  This module is the plain, seeded stand-in that
drives the page table for the stack workload:

  every ``commit_every`` steps (step 8j, j = 1..7) the byte target is
  (1 - 0.6 * j / 7) * F8, F8 = sum_i M_i^8; the block with the lowest
  accumulated routing mass among those with q > seed (ties by layer, expert,
  then down before gate_up) is lowered by one bit, repeatedly, until
  sum_i M_i^{q_i} <= target or no block can be lowered.

The function is pure host logic over plain numbers, so it is tested on the CPU;
the GPU supplies the routing-mass numerators (pw_moe_route_topk) and the page
table executes the commits.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Sequence, Tuple

GATE_UP, DOWN = 0, 1


def byte_target(step: int, commit_every: int, n_commits: int, f8: int, final_fraction: float = 0.4) -> int:
    """Target bytes after the commit at ``step`` (a multiple of commit_every)."""
    j = step // commit_every
    j = max(0, min(j, n_commits))
    return int((1.0 - (1.0 - final_fraction) * j / n_commits) * f8)


def plan_lowering(bits: Dict[Tuple[int, int, int], int], mass: Dict[Tuple[int, int], float],
                  block_bytes: Callable[[Tuple[int, int, int], int], int], seed_bits: int, target: int
                  ) -> List[Tuple[Tuple[int, int, int], int, int]]:
    """Greedy lowering.  ``bits`` maps (layer, expert, u) -> committed q;
    ``mass`` maps (layer, expert) -> accumulated routing mass; ``block_bytes``
    gives M_i^b.  Returns the list of (block, q_old, q_new) steps, one bit at
    a time, in order.  ``bits`` is not modified."""
    q = dict(bits)
    total = sum(block_bytes(b, qb) for b, qb in q.items())
    steps: List[Tuple[Tuple[int, int, int], int, int]] = []

    def key(b):
        layer, expert, u = b
        return (mass.get((layer, expert), 0.0), layer, expert, 0 if u == DOWN else 1)

    order = sorted(q, key=key)
    for b in order:
        while total > target and q[b] > seed_bits:
            old = q[b]
            total -= block_bytes(b, old) - block_bytes(b, old - 1)
            q[b] = old - 1
            steps.append((b, old, old - 1))
        if total <= target:
            break
    return steps


class StackSchedule:
    """Drives one APLMoEStack through the stack workload's commits."""

    def __init__(self, layers: int, experts: int, seed_bits: int, parent_bits: int,
                 block_bytes: Callable[[Tuple[int, int, int], int], int], commit_every: int = 8,
                 n_commits: int = 7, final_fraction: float = 0.4):
        self.L, self.E, self.S, self.P = layers, experts, seed_bits, parent_bits
        self.block_bytes = block_bytes
        self.commit_every, self.n_commits, self.final_fraction = commit_every, n_commits, final_fraction
        self.bits = {(l, e, u): parent_bits for l in range(layers) for e in range(experts) for u in (GATE_UP, DOWN)}
        self.f8 = sum(block_bytes(b, parent_bits) for b in self.bits)

    def resident_bytes(self) -> int:
        return sum(self.block_bytes(b, q) for b, q in self.bits.items())

    def at_boundary(self, step: int, mass_numerators: Sequence[Sequence[float]]
                    ) -> List[Tuple[Tuple[int, int, int], int, int]]:
        """Called after ``step`` steps.  Returns the lowering steps to commit
        now (empty between commit points) and updates the planned bits."""
        if step == 0 or step % self.commit_every or step // self.commit_every > self.n_commits:
            return []
        mass = {(l, e): float(mass_numerators[l][e]) for l in range(self.L) for e in range(self.E)}
        target = byte_target(step, self.commit_every, self.n_commits, self.f8, self.final_fraction)
        plan = plan_lowering(self.bits, mass, self.block_bytes, self.S, target)
        for b, _, new in plan:
            self.bits[b] = new
        return plan


# ---------------------------------------------------------------------------
# GPU driver of the stack workload (torch plumbing around the libpw calls)
# ---------------------------------------------------------------------------
class StackRun:
    """L independent MoE layers on one GPU, stepped with fresh seeded inputs;
    every ``commit_every`` steps the schedule lowers blocks and the released
    plane/LUT tensors are dropped (their memory returns to the caching
    allocator for later allocations on the stream).

    With ``offload=True`` lowering follows §3.3's offload instead: the pages
    above the new bitwidth are first copied to pinned host memory on a copy
    stream (overlapping the next layer calls), q_i drops at once, and each
    page's GPU buffer is dropped by the first step boundary whose poll sees its
    copy finish.  Host buffers are slices of one pinned arena sized for every
    page the schedule can lower (allocated up front, outside any timing)."""

    def __init__(self, wl, device, layers=None, commit_every: int = 8, n_commits: int = 7,
                 final_fraction: float = 0.4, offload: bool = False, batched: bool = False):
        from . import synth
        from .layer import APLMoEStack, MoECall, MoELayersCall, load_layer
        import torch
        self.torch, self.synth = torch, synth
        self.wl = wl
        self.L = wl.layers if layers is None else layers
        sh = wl.shape
        self.stack = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, self.L, wl.parent_bits,
                                 wl.seed_bits, device)
        for layer in range(self.L):
            li = synth.layer_inputs(wl, layer=layer, device=device)
            load_layer(self.stack, layer, li)
            del li
        self.stack.sync()
        self.call = MoECall(self.stack, wl.tokens)
        # batched: every layer of a step in one launch (pw_moe_route_apl_ffn_layers)
        self.layers_call = MoELayersCall(self.stack, wl.tokens, self.L) if batched else None

        def block_bytes(b, q):
            return self.stack.block_bytes_at(self.stack.block_id(*b), q)
        self.schedule = StackSchedule(self.L, sh.experts, wl.seed_bits, wl.parent_bits, block_bytes,
                                      commit_every, n_commits, final_fraction)
        self.step_no = 0
        self.offload = offload
        self.offloaded_bytes = 0
        if offload:
            st = self.stack
            arena = sum(st.block_bytes_at(b, st.P) - st.block_bytes_at(b, st.S) for b in range(st.n_blocks))
            self.arena = torch.empty(arena + 256 * 2 * st.P * st.n_blocks, dtype=torch.uint8, pin_memory=True)
            self.arena_used = 0
            self.copy_stream = torch.cuda.Stream(device=st.device)
            st.host_alloc = self._host_slice

    def inputs(self, layer: int, step: int):
        dev = self.stack.device
        return (self.synth.activations(self.wl, layer, step, dev),
                self.synth.router_logits(self.wl, layer, step, dev))

    def inputs_all(self, step: int):
        """Every layer's inputs of a step, stacked: x [L][T][H], logits [L][T][E]."""
        xs, lgs = zip(*(self.inputs(layer, step) for layer in range(self.L)))
        return self.torch.stack(xs).contiguous(), self.torch.stack(lgs).contiguous()

    def step(self, xs=None, logits=None, on_layer=None):
        """One step: every layer routes and runs its fused expert layer (one
        launch per layer, or one launch for all layers when batched), then
        the step boundary commits any lowering due.  ``on_layer(layer, y)`` is
        called after each layer's output is enqueued (per-layer calls reuse
        ``y`` for the next layer).  Batched steps take ``xs`` / ``logits`` as
        stacked [L][T][...] tensors."""
        if self.layers_call is not None:
            if xs is None:
                xs, logits = self.inputs_all(self.step_no)
            y = self.layers_call(0, xs, logits, mass=self.call.mass)
            if on_layer is not None:
                for layer in range(self.L):
                    on_layer(layer, y[layer])
        else:
            for layer in range(self.L):
                x, lg = (xs[layer], logits[layer]) if xs is not None else self.inputs(layer, self.step_no)
                y = self.call(layer, x, lg)
                if on_layer is not None:
                    on_layer(layer, y)
        self.step_no += 1
        return self.boundary()

    def status(self) -> int:
        """The device status word of the calls (0 = fine)."""
        st = int(self.call.status.item())
        if st == 0 and self.layers_call is not None:
            st = int(self.layers_call.status.item())
        return st

    def _host_slice(self, nbytes: int):
        start = (self.arena_used + 255) & ~255
        if start + nbytes > self.arena.numel():
            raise RuntimeError("stack offload: host arena exhausted")
        self.arena_used = start + nbytes
        return self.arena[start:start + nbytes]

    def boundary(self):
        """Commit the schedule's lowering at a step boundary; returns the
        (block, q_old, q_new) steps committed and the bytes released."""
        if self.offload:
            self.stack.poll()      # drop GPU pages whose offload copy has finished
        if self.step_no % self.schedule.commit_every:
            return [], 0
        mass = self.call.mass.float().cpu().tolist()    # routing-mass numerators (Eq. 1)
        plan = self.schedule.at_boundary(self.step_no, mass)
        released = 0
        for (layer, e, u), _, new in plan:
            b = self.stack.block_id(layer, e, u)
            if self.offload:
                before = self.stack.host_bytes
                released += self.stack.offload(b, new, self.copy_stream)
                self.offloaded_bytes += self.stack.host_bytes - before
            else:
                released += self.stack.commit(b, new)
        if plan:
            self.stack.sync()
        return plan, released

    def finish_offloads(self, limit_s: float = 60.0) -> None:
        """Wait (host side) until every offload copy finished and its GPU pages
        were dropped."""
        import time
        t0 = time.time()
        while self.stack.poll() > 0:
            if time.time() - t0 > limit_s:
                raise RuntimeError("page copies did not finish")
            time.sleep(0.001)
