"""Plain float64 CPU oracle (test infrastructure only; see oracle/__init__.py).

Citations name the arXiv text of "PagedWeight: Efficient MoE LLM Serving with
Dynamic Quality-Aware Weight Quantization" by section, equation and figure.

Everything here is deliberately slow and literal: no blocking, no fusion, no
reordering beyond what the definitions state.  Large blocks are processed in
row chunks only to bound host memory; chunking rows does not change any sum.

Storage format read and written by this oracle (the pages fix the overlay
semantics but not the memory layout; this is the library's documented
"tiled" layout, written out independently here):

  A block W has N rows and K columns of P-bit parent indices idx[n][j].
  It is stored as P separate bit-planes.  Plane p (p = 0 is the most
  significant) holds bit P-1-p of every index, so the b-bit index of the
  overlay is the top b bits: idx_b = idx >> (P - b)  (§1; Figure 3 draws the
  planes b7 ... b0 and the caption says subsets of planes give the lower
  bitwidths).  Requires N % 128 == 0 and K % 128 == 0.  A plane has N*K/8 bytes.

  Bit (n, j) of a plane sits at this position:
    half  = n // (N/2);  r = n % (N/2);  strip = r // 64;  rr = r % 64
    w     = rr // 16;    i = rr % 16 + 16*half;  pos = 32*w + i
    tile  = j // 128;    jj = j % 128;   word = jj // 32;  t = jj % 32
    bit   = 4*(t % 8) + t // 8                (bit of a little-endian uint32)
    byte offset of that uint32 = (strip * (K/128) + tile) * 2048 + 16*pos + 4*word

  The LUT of bitwidth b (fp16 [N][2^b], one row of centroids per output row,
  Figure 3 caption) is stored "tiled" too: with strip, w and i of row n as
  above, entry c of row n sits at byte
    (strip * 2^b + c) * 256 + 4*((w % 2)*32 + i) + 2*(w // 2)
  so the table of a 128-row strip is one contiguous run of 2^b * 256 bytes.
"""
from __future__ import annotations

import math
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

TILE_ROWS = 128
TILE_COLS = 128
TILE_BYTES = 2048

GATE_UP = 0
DOWN = 1


# ----------------------------------------------------------------------------
# Bit-plane layout
# ----------------------------------------------------------------------------
def check_block_shape(N: int, K: int) -> None:
    if N <= 0 or K <= 0 or N % TILE_ROWS or K % TILE_COLS:
        raise ValueError(f"block {N}x{K}: rows and cols must be multiples of 128")


def plane_bytes(N: int, K: int) -> int:
    check_block_shape(N, K)
    return N * K // 8


def bit_address(n, j, N: int, K: int):
    """Linear bit address (8 * byte + bit-in-byte) of element (n, j) inside a
    plane; n and j broadcast like numpy arrays.  Follows the layout in the
    module docstring literally."""
    n = np.asarray(n, dtype=np.int64)
    j = np.asarray(j, dtype=np.int64)
    half_rows = N // 2
    half = n // half_rows
    r = n % half_rows
    strip = r // 64
    rr = r % 64
    w = rr // 16
    i = rr % 16 + 16 * half
    pos = 32 * w + i
    tile = j // TILE_COLS
    jj = j % TILE_COLS
    word = jj // 32
    t = jj % 32
    bit = 4 * (t % 8) + t // 8
    word_byte = (strip * (K // TILE_COLS) + tile) * TILE_BYTES + 16 * pos + 4 * word
    # little-endian uint32: bit b of the word is bit b % 8 of byte b // 8
    return 8 * word_byte + bit


def lut_tiled_offset(n, c, N: int, b: int):
    """Byte offset of LUT entry c of row n in the tiled LUT layout (module
    docstring); n and c broadcast like numpy arrays."""
    n = np.asarray(n, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    half_rows = N // 2
    half = n // half_rows
    r = n % half_rows
    strip = r // 64
    rr = r % 64
    w = rr // 16
    i = rr % 16 + 16 * half
    return (strip * (1 << b) + c) * 256 + 4 * ((w % 2) * 32 + i) + 2 * (w // 2)


def pack_lut_tiled(lut: np.ndarray) -> np.ndarray:
    """fp16 [N][2^b] row-major LUT -> uint8 bytes in the tiled LUT layout."""
    lut = np.asarray(lut, dtype=np.float16)
    N, C = lut.shape
    b = C.bit_length() - 1
    if C != 1 << b or N % TILE_ROWS:
        raise ValueError("LUT must be [N][2^b] with N % 128 == 0")
    out = np.zeros(N * C * 2, dtype=np.uint8)
    off = lut_tiled_offset(np.arange(N)[:, None], np.arange(C)[None, :], N, b).ravel()
    raw = lut.view(np.uint8).reshape(N * C, 2)
    out[off] = raw[:, 0]
    out[off + 1] = raw[:, 1]
    return out


def pack_bitplanes(idx: np.ndarray, parent_bits: int) -> List[np.ndarray]:
    """Parent indices uint8 [N][K] -> ``parent_bits`` planes, MSB plane first,
    each a uint8 array of N*K/8 bytes in the tiled layout."""
    idx = np.asarray(idx)
    N, K = idx.shape
    check_block_shape(N, K)
    if idx.size and int(idx.max()) >= (1 << parent_bits):
        raise ValueError("index exceeds parent bitwidth")
    addr = bit_address(np.arange(N)[:, None], np.arange(K)[None, :], N, K).ravel()
    planes = []
    for p in range(parent_bits):
        bits = np.zeros(N * K, dtype=np.uint8)
        bits[addr] = ((idx.astype(np.int64) >> (parent_bits - 1 - p)) & 1).ravel()
        planes.append(np.packbits(bits, bitorder="little"))
    return planes


def unpack_indices(planes: Sequence[np.ndarray], b: int, N: int, K: int,
                   rows: Optional[Tuple[int, int]] = None) -> np.ndarray:
    """The b-bit overlay index of rows [r0, r1): idx_b = sum_{p<b} bit_p << (b-1-p)
    using only the top b planes (§1, Figure 3 caption).  int64 [r1-r0][K]."""
    check_block_shape(N, K)
    if b < 1 or b > len(planes):
        raise ValueError("bitwidth outside the planes given")
    r0, r1 = rows if rows is not None else (0, N)
    addr = bit_address(np.arange(r0, r1)[:, None], np.arange(K)[None, :], N, K)
    # only unpack the bytes of the strips these rows live in (bounds host memory)
    strip_bits = (K // TILE_COLS) * TILE_BYTES * 8
    lo = int(addr.min()) // strip_bits * strip_bits if addr.size else 0
    hi = (int(addr.max()) // strip_bits + 1) * strip_bits if addr.size else 0
    out = np.zeros((r1 - r0, K), dtype=np.int64)
    for p in range(b):
        seg = np.asarray(planes[p], dtype=np.uint8)[lo // 8: hi // 8]
        bits = np.unpackbits(seg, bitorder="little")
        out += bits[addr - lo].astype(np.int64) << (b - 1 - p)
    return out


# ----------------------------------------------------------------------------
# Dequantisation and the any-precision linear map
# ----------------------------------------------------------------------------
def dequant(idx_b: np.ndarray, lut_b: np.ndarray, rows: Optional[Tuple[int, int]] = None) -> np.ndarray:
    """W[n][j] = LUT_b[n][idx_b[n][j]] in float64 (Figure 3 caption: each bitwidth
    has its own table of centroids; one LUT row per output row)."""
    lut = np.asarray(lut_b).astype(np.float64)
    r0, r1 = rows if rows is not None else (0, lut.shape[0])
    return np.take_along_axis(lut[r0:r1], idx_b, axis=1)


def apl_linear(planes: Sequence[np.ndarray], lut_b: np.ndarray, b: int, N: int, K: int,
               x: np.ndarray, row_chunk: int = 2048) -> np.ndarray:
    """out[m][n] = sum_j W_b[n][j] * x[m][j]  with W_b dequantised at bitwidth b.
    x is [M][K]; returns float64 [M][N]."""
    xm = np.asarray(x).astype(np.float64)
    out = np.zeros((xm.shape[0], N), dtype=np.float64)
    for r0 in range(0, N, row_chunk):
        r1 = min(N, r0 + row_chunk)
        W = dequant(unpack_indices(planes, b, N, K, (r0, r1)), lut_b, (r0, r1))
        out[:, r0:r1] = xm @ W.T
    return out


# ----------------------------------------------------------------------------
# Routing (§2.1, Eq. 1)
# ----------------------------------------------------------------------------
def route_topk(logits: np.ndarray, k: int) -> Dict[str, np.ndarray]:
    """Top-k routing of fp32 logits [T][E].

    softmax over all E experts in float64; the k experts with the largest
    logit are chosen one at a time (ties go to the lower expert index), and
    their probabilities are renormalised over the k choices.  The assignment
    slots s = t*k + j are ordered by (expert, token, j); offsets[e] is the
    first position of expert e.  Routing mass is Eq. 1: the routing weight an
    expert received over all tokens and choices, over the total weight.
    """
    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    z = lg.astype(np.float64)
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ids = np.zeros((T, k), dtype=np.int32)
    for t in range(T):
        taken = np.zeros(E, dtype=bool)
        for j in range(k):
            best = -1
            for e in range(E):
                if taken[e]:
                    continue
                if best < 0 or lg[t, e] > lg[t, best]:
                    best = e
            ids[t, j] = best
            taken[best] = True
    psel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    w = psel / psel.sum(axis=1, keepdims=True)
    # counting sort of the slots by expert, keeping (token, j) order
    A = T * k
    counts = np.zeros(E, dtype=np.int64)
    for s in range(A):
        counts[ids[s // k, s % k]] += 1
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    cursor = offsets[:-1].astype(np.int64).copy()
    perm = np.zeros(A, dtype=np.int32)
    inv_perm = np.zeros(A, dtype=np.int32)
    for s in range(A):
        e = ids[s // k, s % k]
        perm[cursor[e]] = s
        inv_perm[s] = cursor[e]
        cursor[e] += 1
    # Eq. 1: m_e = sum_t sum_k r 1{z = e} / sum_t sum_k r
    mass = np.zeros(E, dtype=np.float64)
    for t in range(T):
        for j in range(k):
            mass[ids[t, j]] += w[t, j]
    total = w.sum()
    if total > 0:
        mass /= total
    return dict(ids=ids, w=w, offsets=offsets, perm=perm, inv_perm=inv_perm, mass=mass,
                probs=p)


def route_topk_shared(logits: np.ndarray, k: int, S: int) -> Dict[str, np.ndarray]:
    """Top-k routing plus S shared experts.

    The pages' Table 1 lists models with shared experts (60 routed + 4 shared,
    top-4; 128 routed + 1 shared, top-8) and gives them no gate; the reading
    here: every token also passes through the shared experts E .. E+S-1 with
    weight 1, added to its routed output.  Each token has K = k + S slots
    (its routed picks, as route_topk, then the shared experts); slots
    s = t*K + j are ordered by (expert, token, j) over E + S experts; mass is
    Eq. 1 over all E + S experts.
    """
    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    if S < 0:
        raise ValueError("need S >= 0")
    r = route_topk(lg, k)
    K = k + S
    ids = np.concatenate([r["ids"], np.tile(E + np.arange(S, dtype=np.int32), (T, 1))], axis=1).astype(np.int32)
    w = np.concatenate([r["w"], np.ones((T, S), dtype=np.float64)], axis=1)
    expert_of_slot = ids.reshape(-1).astype(np.int64)              # slot order is (token, j)
    perm = np.argsort(expert_of_slot, kind="stable").astype(np.int32)
    inv_perm = np.empty(T * K, dtype=np.int32)
    inv_perm[perm] = np.arange(T * K, dtype=np.int32)
    counts = np.bincount(expert_of_slot, minlength=E + S)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    mass = np.zeros(E + S, dtype=np.float64)
    np.add.at(mass, expert_of_slot, w.reshape(-1))
    total = w.sum()
    if total > 0:
        mass /= total
    return dict(ids=ids, w=w, offsets=offsets, perm=perm, inv_perm=inv_perm, mass=mass)


# ----------------------------------------------------------------------------
# The MoE layer (§3.3: routing, the routed experts' two projections and the weighted sum)
# ----------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


class Block:
    """One linear-block (layer, expert, u) as the oracle sees it: its planes,
    its LUTs by bitwidth and the committed bitwidth q."""

    def __init__(self, planes: Sequence[np.ndarray], luts: Dict[int, np.ndarray], q: int,
                 N: int, K: int):
        self.planes, self.luts, self.q, self.N, self.K = list(planes), luts, int(q), N, K

    def linear(self, x: np.ndarray) -> np.ndarray:
        """[M][K] -> [M][N] at the committed bitwidth."""
        return apl_linear(self.planes, self.luts[self.q], self.q, self.N, self.K, x)


class IndexBlock:
    """A linear-block given by its parent indices instead of its planes: the
    q-bit index is the definition idx >> (P - q) (the overlay rule, §1).  Equal
    to Block on packed planes by the overlay pin; used where packing a large
    block on the host would dominate the test time."""

    def __init__(self, idx: np.ndarray, luts: Dict[int, np.ndarray], q: int, parent_bits: int):
        self.idx, self.luts, self.q, self.P = idx, luts, int(q), int(parent_bits)
        self.N, self.K = idx.shape

    def linear(self, x: np.ndarray, row_chunk: int = 2048) -> np.ndarray:
        xm = np.asarray(x).astype(np.float64)
        out = np.zeros((xm.shape[0], self.N), dtype=np.float64)
        for r0 in range(0, self.N, row_chunk):
            r1 = min(self.N, r0 + row_chunk)
            idx_b = self.idx[r0:r1].astype(np.int64) >> (self.P - self.q)
            W = dequant(idx_b, self.luts[self.q], (r0, r1))
            out[:, r0:r1] = xm @ W.T
        return out


def moe_layer(x: np.ndarray, ids: np.ndarray, w: np.ndarray, I: int,
              blocks: Callable[[int, int], Block], tokens: Optional[Sequence[int]] = None
              ) -> np.ndarray:
    """y[t] = sum_j w[t][j] * down_e( silu(gate_e x_t) * up_e x_t ),  e = ids[t][j].

    gate_up rows [0, I) are the gate, rows [I, 2I) the up projection; the
    routing weight is applied after the down projection, in the output
    accumulation.  ``blocks(e, u)`` returns the Block of expert e.  ``tokens``
    restricts the output to a subset of tokens (others stay zero); a negative
    expert id leaves that assignment out (used to time a subset of experts).
    Returns float64 [T][H].
    """
    xm = np.asarray(x).astype(np.float64)
    T = xm.shape[0]
    k = ids.shape[1]
    want = np.ones(T, dtype=bool) if tokens is None else np.isin(np.arange(T), tokens)
    H = xm.shape[1]
    y = np.zeros((T, H), dtype=np.float64)
    experts = sorted(set(int(e) for e in ids[want].ravel() if e >= 0))
    for e in experts:
        tt, jj = np.nonzero((ids == e) & want[:, None])
        if tt.size == 0:
            continue
        G = blocks(e, GATE_UP).linear(xm[tt])          # [n][2I]
        h = silu(G[:, :I]) * G[:, I:]                    # [n][I]
        D = blocks(e, DOWN).linear(h)                    # [n][H]
        for i in range(tt.size):
            y[tt[i]] += w[tt[i], jj[i]] * D[i]
    return y


# ----------------------------------------------------------------------------
# Page accounting (§3.1, Eq. 3)
# ----------------------------------------------------------------------------
def page_bytes(N: int, K: int, seed_bits: int, b: int) -> int:
    """M_i^b: bytes a block needs on the GPU at bitwidth b -- the top b planes
    plus the LUTs of every supported bitwidth up to b (so that lowering needs
    no transfer).  fp16 LUT entries."""
    if b < seed_bits:
        raise ValueError("below the seed bitwidth")
    return b * N * K // 8 + sum(N * (1 << kk) * 2 for kk in range(seed_bits, b + 1))


def released_bytes(N: int, K: int, seed_bits: int, b: int, b_new: int) -> int:
    """Eq. 3: Delta^{b -> b'} = M^b - M^{b'} for b' < b."""
    if not b_new < b:
        raise ValueError("Eq. 3 is defined for b' < b")
    return page_bytes(N, K, seed_bits, b) - page_bytes(N, K, seed_bits, b_new)


def compare(y_ref: np.ndarray, y: np.ndarray) -> Dict[str, float]:
    """rel-L2 error and max-abs error relative to rms(y_ref)."""
    y_ref = np.asarray(y_ref, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    diff = y - y_ref
    nref = float(np.linalg.norm(y_ref))
    rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    return dict(rel_l2=float(np.linalg.norm(diff)) / nref if nref > 0 else float(np.linalg.norm(diff)),
                max_abs=float(np.max(np.abs(diff))) if diff.size else 0.0,
                rms=rms,
                max_abs_over_rms=(float(np.max(np.abs(diff))) / rms) if rms > 0 and diff.size else 0.0)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("annotations", "math", "np")]
