"""Device storage and call plumbing for Any-Precision MoE layers on one GPU.

PyTorch is used here only for device memory and streams: every computation
(packing, routing, the fused expert layer) is a libpw kernel called through
the C ABI binding in ``pw.py``.

``APLMoEStack`` owns, for L MoE layers of E experts, the bit-plane tensors and
LUT tensors of every per-expert linear-block (layer, expert, gate_up|down),
the libpw page table that borrows them, and the device descriptor array the
fused kernel reads.  Lowering a block's committed bitwidth drops the plane and
LUT tensors above it (the torch caching allocator reuses that memory for
later allocations on the same stream, i.e. after the launches already
enqueued -- the "release at a safe boundary" of §3.3 of the PagedWeight
arXiv text).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Dict, List, Optional

import torch

from . import pw

GATE_UP, DOWN = 0, 1


class APLMoEStack:
    def __init__(self, hidden: int, intermediate: int, experts: int, top_k: int, layers: int = 1,
                 parent_bits: int = 8, seed_bits: int = 3, device="cuda", shared: int = 0):
        # E counts every expert with blocks (routed, then `shared` shared
        # experts that every token passes through with weight 1); k is the
        # routed top-k
        self.H, self.I, self.E, self.k, self.L = hidden, intermediate, experts + shared, top_k, layers
        self.routed, self.shared = experts, shared
        self.P, self.S = parent_bits, seed_bits
        self.device = torch.device(device)
        self.n_blocks = layers * self.E * 2
        infos = []
        for b in range(self.n_blocks):
            rows, cols = self.block_shape(b % 2)
            infos.append(pw.pw_block_info(rows, cols, parent_bits, seed_bits, pw.PW_LAYOUT_TILED, 0))
        self.table = pw.pw_page_table_create(infos)
        self.planes: Dict[int, List[Optional[torch.Tensor]]] = {}
        self.luts: Dict[int, Dict[int, torch.Tensor]] = {}
        self.host: Dict[tuple, torch.Tensor] = {}   # (block, page) -> pinned host copy
        self.host_bytes = 0                          # bytes of host copies started
        self.host_alloc = lambda n: torch.empty(n, dtype=torch.uint8, pin_memory=True)
        self._moving = set()                         # blocks with transfers started since the last poll
        nbytes = pw.pw_desc_bytes(self.n_blocks)
        self.desc = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)

    def __del__(self):
        t = getattr(self, "table", None)
        if t is not None:
            try:
                pw.pw_page_table_destroy(t)
            except Exception:
                pass
            self.table = None

    # ------------------------------------------------------------------
    def block_shape(self, u: int):
        return (2 * self.I, self.H) if u == GATE_UP else (self.H, self.I)

    def block_id(self, layer: int, expert: int, u: int) -> int:
        return (layer * self.E + expert) * 2 + u

    def load_block(self, block: int, idx: torch.Tensor, luts: Dict[int, torch.Tensor], q: int,
                   keep_planes: Optional[int] = None, stream=None) -> None:
        """Pack parent indices (uint8 [rows][cols] on the device) into P planes,
        keep the top ``keep_planes`` (default q) and the LUTs seed..keep
        (row-major fp16, stored in the tiled LUT layout), attach them to the
        page table and commit q."""
        rows, cols = self.block_shape(block % 2)
        assert tuple(idx.shape) == (rows, cols)
        keep = q if keep_planes is None else keep_planes
        nb = pw.pw_plane_bytes(rows, cols)
        planes = [torch.empty(nb // 4, dtype=torch.int32, device=self.device) for _ in range(self.P)]
        pw.pw_pack_bitplanes(idx.to(self.device).contiguous(), self.P, planes, stream=stream)
        kept: List[Optional[torch.Tensor]] = [planes[p] if p < keep else None for p in range(self.P)]
        del planes
        self.planes[block] = kept
        self.luts[block] = {}
        for p in range(keep):
            pw.pw_page_table_attach_plane(self.table, block, p, kept[p].data_ptr())
        for b in range(self.S, keep + 1):
            t = luts[b].to(self.device).contiguous()
            assert t.dtype == torch.float16 and tuple(t.shape) == (rows, 1 << b)
            tiled = torch.empty_like(t)
            pw.pw_pack_lut(t, tiled, stream=stream)     # LUT pages are stored in the tiled LUT layout
            self.luts[block][b] = tiled
            pw.pw_page_table_attach_lut(self.table, block, b, tiled.data_ptr())
        self.commit(block, q)

    def commit(self, block: int, q: int) -> int:
        """Commit q for a block; returns the bytes released (Eq. 3)."""
        before = self.resident_bytes_of(block)
        mask = pw.pw_page_table_set_bits(self.table, block, q)
        for p in range(self.P):
            if mask >> p & 1:
                self.planes[block][p] = None
        for b in range(self.S, self.P + 1):
            if mask >> (8 + b) & 1:
                self.luts[block].pop(b, None)
        return before - self.resident_bytes_of(block)

    # -- asynchronous page movement (§3.3, Figure 4) -------------------------
    def pages_between(self, block: int, lo: int, hi: int) -> List[int]:
        """Page ids a block holds at bitwidth hi but not at lo: planes lo..hi-1
        and the LUTs of bitwidths lo+1..hi."""
        return list(range(lo, hi)) + [pw.PW_PAGE_LUT(b) for b in range(max(lo + 1, self.S), hi + 1)]

    def offload(self, block: int, q: int, copy_stream: torch.cuda.Stream) -> int:
        """Lower a block to q keeping host copies of the pages above q: start
        copying each of them to pinned host memory on `copy_stream`, then commit
        q.  Pages whose copy is still running stay on the GPU until a later
        poll() sees the copy finish.  Returns the bytes the commit releases
        (Eq. 3)."""
        cur = self.committed_bits(block)
        copy_stream.wait_stream(torch.cuda.current_stream(self.device))
        for page in self.pages_between(block, q, cur):
            st, _, _ = pw.pw_page_state(self.table, block, page)
            if not st & pw.PW_PAGE_GPU or st & pw.PW_PAGE_CPU:
                continue
            host = self.host.get((block, page))
            if host is None:
                host = self.host_alloc(pw.pw_page_bytes(self.table, block, page))
                self.host[(block, page)] = host
            pw.pw_page_offload(self.table, block, page, host, stream=copy_stream)
            self.host_bytes += pw.pw_page_bytes(self.table, block, page)
            self._moving.add(block)
        return self.commit(block, q)

    def reload(self, block: int, q: int, copy_stream: torch.cuda.Stream) -> None:
        """Start restoring a block's pages up to bitwidth q from their host
        copies into new device buffers on `copy_stream`; raise_to(q) succeeds
        once poll() has seen every copy finish."""
        cur = self.committed_bits(block)
        for page in self.pages_between(block, cur, q):
            st, _, _ = pw.pw_page_state(self.table, block, page)
            if st & (pw.PW_PAGE_GPU | pw.PW_PAGE_TO_GPU):
                continue
            dev = torch.empty(pw.pw_page_bytes(self.table, block, page), dtype=torch.uint8, device=self.device)
            dev.record_stream(copy_stream)
            pw.pw_page_reload(self.table, block, page, None, dev, stream=copy_stream)
            self._moving.add(block)
            if page < pw.PW_MAX_BITS:
                self.planes[block][page] = dev
            else:
                self.luts[block][page - pw.PW_MAX_BITS] = dev

    def poll(self) -> int:
        """Advance finished page transfers and drop the device buffers of pages
        the table retired after their offload copy; returns the transfers
        still running."""
        n = pw.pw_page_table_poll(self.table)
        for block in sorted(self._moving):
            m = pw.pw_page_table_take_released(self.table, block)
            for p in range(self.P):
                if m >> p & 1:
                    self.planes[block][p] = None
            for b in range(self.S, self.P + 1):
                if m >> (8 + b) & 1:
                    self.luts[block].pop(b, None)
        if n == 0:
            self._moving.clear()
        return n

    def raise_to(self, block: int, q: int) -> bool:
        """Commit a higher bitwidth if its pages are GPU-resident (after
        reload() and a poll() that saw the copies finish); False otherwise."""
        try:
            self.commit(block, q)
            return True
        except pw.PwError as e:
            if e.code == pw.PW_ERR_NOT_RESIDENT:
                return False
            raise

    def block_bytes_at(self, block: int, q: int) -> int:
        """M_i^q of Eq. 3 for a block (page-table arithmetic)."""
        return pw.pw_page_table_bytes(self.table, block, q)

    def resident_bytes_of(self, block: int) -> int:
        q, _, _ = pw.pw_page_table_get(self.table, block)
        return pw.pw_page_table_bytes(self.table, block, q) if q > 0 else 0

    def committed_bits(self, block: int) -> int:
        return pw.pw_page_table_get(self.table, block)[0]

    def resident_bytes(self) -> int:
        return pw.pw_page_table_resident_bytes(self.table)

    def sync(self, stream=None) -> None:
        pw.pw_page_table_sync(self.table, self.desc, stream=stream)


@dataclass
class RouteBuffers:
    ids: torch.Tensor
    w: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    inv_perm: torch.Tensor


class MoECall:
    """Preallocated buffers for one (T, shape) and the layer call: routing and
    the fused expert layer in one launch (pw_moe_route_apl_ffn), or with
    ``fused=False`` as two launches, pw_moe_route_topk then pw_moe_apl_ffn."""

    def __init__(self, stack: APLMoEStack, tokens: int, device=None, fused: bool = True):
        dev = stack.device if device is None else torch.device(device)
        T, E, k = tokens, stack.E, stack.k + stack.shared   # all experts, slots per token
        self.stack, self.T, self.fused = stack, T, fused
        A = max(1, T * k)
        self.route = RouteBuffers(
            ids=torch.empty((max(T, 1), k), dtype=torch.int32, device=dev),
            w=torch.empty((max(T, 1), k), dtype=torch.float32, device=dev),
            offsets=torch.empty((E + 1,), dtype=torch.int32, device=dev),
            perm=torch.empty((A,), dtype=torch.int32, device=dev),
            inv_perm=torch.empty((A,), dtype=torch.int32, device=dev))
        self.mass = torch.zeros((stack.L, E), dtype=torch.float32, device=dev)
        ws = pw.pw_moe_apl_ffn_workspace(T, stack.H, stack.I, E, k)
        self.ws = torch.empty((max(ws, 256),), dtype=torch.uint8, device=dev)
        self.y = torch.empty((max(T, 1), stack.H), dtype=torch.float16, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)

    def __call__(self, layer: int, x: torch.Tensor, logits: torch.Tensor, options=None, stream=None,
                 accumulate_mass: bool = True) -> torch.Tensor:
        s, r = self.stack, self.route
        mass = self.mass[layer] if accumulate_mass else None
        if self.fused:
            if s.shared:
                opts = pw.pw_ffn_options()
                if options is not None:
                    ctypes.memmove(ctypes.addressof(opts), ctypes.addressof(options), ctypes.sizeof(opts))
                opts.shared_experts = s.shared
                options = opts
            pw.pw_moe_route_apl_ffn(s.desc, layer, x, logits, s.I, s.routed, s.k, r.ids, r.w, r.offsets, r.perm,
                                    r.inv_perm, mass, self.ws, self.y, self.status, options=options, stream=stream)
        else:
            pw.pw_moe_route_topk_shared(logits, s.k, s.shared, r.ids, r.w, r.offsets, r.perm, r.inv_perm, mass,
                                        stream=stream)
            pw.pw_moe_apl_ffn(s.desc, layer, x, s.I, s.E, s.k + s.shared, r.ids, r.w, r.offsets, r.perm,
                              r.inv_perm, self.ws, self.y, self.status, options=options, stream=stream)
        return self.y[: self.T]


class MoELayersCall:
    """Preallocated buffers for ``layers`` consecutive layers of a stack, each
    with ``tokens`` tokens, run in one launch (pw_moe_route_apl_ffn_layers).
    The routing arrays are in the layers' concatenated index space
    (``offsets`` [L*E+1], ``perm``/``inv_perm`` [L*T*k]); ``ids`` and ``w`` are
    [L][T][k] with each layer's own expert ids."""

    def __init__(self, stack: APLMoEStack, tokens: int, layers: int, device=None):
        dev = stack.device if device is None else torch.device(device)
        L, T, E, k = layers, tokens, stack.E, stack.k + stack.shared
        self.stack, self.T, self.L = stack, T, L
        A = max(1, L * T * k)
        self.ids = torch.empty((L, max(T, 1), k), dtype=torch.int32, device=dev)
        self.w = torch.empty((L, max(T, 1), k), dtype=torch.float32, device=dev)
        self.offsets = torch.empty((L * E + 1,), dtype=torch.int32, device=dev)
        self.perm = torch.empty((A,), dtype=torch.int32, device=dev)
        self.inv_perm = torch.empty((A,), dtype=torch.int32, device=dev)
        ws = pw.pw_moe_apl_ffn_workspace(L * T, stack.H, stack.I, L * E, k)
        self.ws = torch.empty((max(ws, 256),), dtype=torch.uint8, device=dev)
        self.y = torch.empty((L, max(T, 1), stack.H), dtype=torch.float16, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)

    def __call__(self, layer0: int, x: torch.Tensor, logits: torch.Tensor, mass: Optional[torch.Tensor] = None,
                 options=None, stream=None) -> torch.Tensor:
        """x [L][T][H], logits [L][T][E_routed]; ``mass`` [L][E] (accumulated)
        or None.  Returns y [L][T][H]."""
        s = self.stack
        opts = pw.pw_ffn_options()
        if options is not None:
            ctypes.memmove(ctypes.addressof(opts), ctypes.addressof(options), ctypes.sizeof(opts))
        opts.shared_experts = s.shared
        pw.pw_moe_route_apl_ffn_layers(s.desc, layer0, x, logits, s.I, s.routed, s.k, self.ids, self.w, self.offsets,
                                       self.perm, self.inv_perm, mass, self.ws, self.y, self.status, options=opts,
                                       stream=stream)
        return self.y[:, : self.T]


def load_layer(stack: APLMoEStack, layer: int, inputs, experts=None, stream=None) -> None:
    """Load one layer's blocks from a synth.LayerInputs-like object (fields
    ``idx[(e, u)]``, ``luts[(e, u)][b]``, ``bits[2e+u]``) at their committed
    bitwidths, keeping only the planes and LUTs those bitwidths need."""
    ex = range(stack.E) if experts is None else experts
    for e in ex:
        for u in (GATE_UP, DOWN):
            stack.load_block(stack.block_id(layer, e, u), inputs.idx[(e, u)], inputs.luts[(e, u)],
                             inputs.bits[2 * e + u], stream=stream)
