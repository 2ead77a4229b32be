"""Pins for the CPU oracle: each checks it against something other than itself.

Citations are to the arXiv text of "PagedWeight: Efficient MoE LLM Serving
with Dynamic Quality-Aware Weight Quantization".  No test here needs a GPU.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import apl

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand_idx(rng, N, K, P):
    return rng.integers(0, 1 << P, size=(N, K), dtype=np.uint8)


# ---------------------------------------------------------------------------
# Layout and overlay (§1; Figure 3 caption)
# ---------------------------------------------------------------------------
def _golden_points():
    pts = []
    with open(os.path.join(HERE, "golden", "layout_points.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            pts.append(tuple(int(v) for v in line.split()))
    return pts


@pytest.mark.parametrize("N,K,n,j,byte,bit", _golden_points())
def test_layout_hand_derived_points(N, K, n, j, byte, bit):
    idx = np.zeros((N, K), dtype=np.uint8)
    idx[n, j] = 1
    (plane,) = apl.pack_bitplanes(idx, 1)
    nz = np.nonzero(plane)[0]
    assert nz.tolist() == [byte]
    assert int(plane[byte]) == 1 << bit


@pytest.mark.parametrize("N,K", [(128, 128), (256, 256), (384, 640), (1024, 128)])
def test_layout_is_a_bijection(N, K):
    n = np.arange(N)[:, None]
    j = np.arange(K)[None, :]
    a = apl.bit_address(n, j, N, K).ravel()
    assert np.array_equal(np.sort(a), np.arange(N * K))


@pytest.mark.parametrize("N,K,P", [(128, 512, 8), (1024, 256, 4), (256, 512, 4), (128, 256, 3)])
def test_overlay_invariant_and_round_trip(N, K, P):
    """For every b: the b-bit index read from the top b planes equals the
    parent index shifted right by P - b; at b = P it is the input."""
    rng = np.random.default_rng(N * 7 + K + P)
    idx = _rand_idx(rng, N, K, P)
    planes = apl.pack_bitplanes(idx, P)
    assert len(planes) == P
    assert all(p.nbytes == N * K // 8 for p in planes)
    for b in range(1, P + 1):
        got = apl.unpack_indices(planes, b, N, K)
        assert np.array_equal(got, idx.astype(np.int64) >> (P - b)), b
    # row-range unpack agrees with the full unpack
    rr = (N // 2 - 8, N // 2 + 8) if N >= 32 else (0, N)
    assert np.array_equal(apl.unpack_indices(planes, P, N, K, rr), idx[rr[0]:rr[1]].astype(np.int64))


def test_lower_planes_do_not_change_higher_bitwidths():
    """Dropping planes >= b leaves the b-bit view untouched (pages above the
    committed bitwidth can be released, §3.1)."""
    rng = np.random.default_rng(5)
    idx = _rand_idx(rng, 128, 512, 8)
    planes = apl.pack_bitplanes(idx, 8)
    for b in range(1, 8):
        assert np.array_equal(apl.unpack_indices(planes[:b], b, 128, 512),
                              apl.unpack_indices(planes, b, 128, 512))


def test_shape_rules():
    with pytest.raises(ValueError):
        apl.pack_bitplanes(np.zeros((64, 256), np.uint8), 4)
    with pytest.raises(ValueError):
        apl.pack_bitplanes(np.zeros((128, 64), np.uint8), 4)
    with pytest.raises(ValueError):
        apl.pack_bitplanes(np.full((128, 128), 16, np.uint8), 4)


# ---------------------------------------------------------------------------
# Dequant + linear: identity LUT and constant LUT
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N,K,P,b,M", [(128, 512, 8, 8, 5), (128, 256, 8, 3, 3), (384, 768, 4, 2, 7)])
def test_identity_lut_is_an_integer_matmul(N, K, P, b, M):
    """LUT_b[n][c] = c makes the layer an exact integer matmul of the b-bit
    indices (sums stay far below 2^53)."""
    rng = np.random.default_rng(N + K + b)
    idx = _rand_idx(rng, N, K, P)
    planes = apl.pack_bitplanes(idx, P)
    lut = np.tile(np.arange(1 << b, dtype=np.float16), (N, 1))
    x = rng.integers(-2, 3, size=(M, K)).astype(np.float16)
    got = apl.apl_linear(planes, lut, b, N, K, x)
    want = x.astype(np.int64) @ (idx.astype(np.int64) >> (P - b)).T
    assert got.shape == (M, N)
    assert np.array_equal(got, want.astype(np.float64))


def test_constant_lut_closed_form():
    """LUT rows constant c_n: out[m][n] = c_n * sum_j x[m][j]."""
    rng = np.random.default_rng(11)
    N, K, P = 128, 512, 6
    idx = _rand_idx(rng, N, K, P)
    planes = apl.pack_bitplanes(idx, P)
    c = (np.arange(N) - 64).astype(np.float16) / np.float16(16)
    lut = np.repeat(c[:, None], 1 << 4, axis=1)
    x = rng.standard_normal((3, K)).astype(np.float16)
    got = apl.apl_linear(planes, lut, 4, N, K, x)
    want = np.outer(x.astype(np.float64).sum(axis=1), c.astype(np.float64))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_lut_row_selects_output_row():
    """Only LUT row n affects output n (one LUT per output row)."""
    rng = np.random.default_rng(12)
    N, K, P = 128, 256, 4
    idx = _rand_idx(rng, N, K, P)
    planes = apl.pack_bitplanes(idx, P)
    lut = np.zeros((N, 16), np.float16)
    lut[5] = np.arange(16)
    x = np.ones((1, K), np.float16)
    out = apl.apl_linear(planes, lut, 4, N, K, x)[0]
    assert np.count_nonzero(out) == 1 and out[5] == idx[5].astype(np.int64).sum()


# ---------------------------------------------------------------------------
# Routing (§2.1, Eq. 1)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,E,k", [(16, 4, 2), (33, 8, 2), (7, 8, 1), (20, 16, 4), (1, 8, 2)])
def test_route_matches_brute_force(T, E, k):
    rng = np.random.default_rng(T * E + k)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    # plant exact ties so the tie-break (lower expert index first) matters
    logits[0, :] = 0.5
    if T > 2:
        logits[2, 1] = logits[2, 3]
    r = apl.route_topk(logits, k)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        assert r["ids"][t].tolist() == order[:k]
        # softmax then renormalise over the k picks == exp over the picks' own sum
        ex = [math.exp(float(logits[t, e]) - float(logits[t].max())) for e in order[:k]]
        s = sum(ex)
        np.testing.assert_allclose(r["w"][t], [v / s for v in ex], rtol=1e-13)
    slots_expert = r["ids"].reshape(-1)
    assert np.array_equal(r["perm"], np.argsort(slots_expert, kind="stable"))
    assert np.array_equal(r["inv_perm"], np.argsort(r["perm"]))
    assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(np.bincount(slots_expert, minlength=E))]))
    np.testing.assert_allclose(r["mass"].sum(), 1.0, rtol=1e-12)
    np.testing.assert_allclose(r["mass"], np.bincount(slots_expert, weights=r["w"].reshape(-1), minlength=E) / T,
                               rtol=1e-12)


def test_route_uniform_pattern_is_balanced():
    """The equal-load logits give every expert exactly A/E assignments."""
    from any_precision_bit_pw_gb300 import synth
    for T in (8, 64, 256):
        lg = synth.router_logits(synth.MIXTRAL_8X7B_SWEEP, tokens=T).numpy()
        r = apl.route_topk(lg, 2)
        assert np.all(np.diff(r["offsets"]) == 2 * T // 8)


# ---------------------------------------------------------------------------
# The whole layer
# ---------------------------------------------------------------------------
def _make_layer(rng, H, I, E, P, bits):
    idx, luts, planes = {}, {}, {}
    for e in range(E):
        for u, (N, K) in ((0, (2 * I, H)), (1, (H, I))):
            idx[e, u] = _rand_idx(rng, N, K, P)
            planes[e, u] = apl.pack_bitplanes(idx[e, u], P)
            luts[e, u] = {b: np.sort((rng.standard_normal((N, 1 << b)) * 0.02).astype(np.float16), axis=1)
                          for b in range(1, P + 1)}
    return idx, luts, planes


def _scalar_layer(x, ids, w, idx, luts, bits, P, H, I, tokens):
    """Pure-Python scalar loops: dequantise straight from the parent index
    (top b bits) and evaluate the layer definition term by term."""
    y = {}
    for t in tokens:
        acc = [0.0] * H
        for j in range(ids.shape[1]):
            e = int(ids[t, j])
            bg, bd = bits[(e, 0)], bits[(e, 1)]
            G = []
            for n in range(2 * I):
                s = 0.0
                row_idx = idx[e, 0][n]
                row_lut = luts[e, 0][bg][n]
                for kk in range(H):
                    s += float(row_lut[int(row_idx[kk]) >> (P - bg)]) * float(x[t, kk])
                G.append(s)
            h = [G[m] / (1.0 + math.exp(-G[m])) * G[I + m] for m in range(I)]
            for n in range(H):
                s = 0.0
                row_idx = idx[e, 1][n]
                row_lut = luts[e, 1][bd][n]
                for m in range(I):
                    s += float(row_lut[int(row_idx[m]) >> (P - bd)]) * h[m]
                acc[n] += float(w[t, j]) * s
        y[t] = acc
    return y


def _oracle_layer(x, r, luts, planes, bits, P, H, I):
    def blocks(e, u):
        N, K = (2 * I, H) if u == 0 else (H, I)
        return apl.Block(planes[e, u], luts[e, u], bits[(e, u)], N, K)
    return apl.moe_layer(x, r["ids"], r["w"], I, blocks)


def test_layer_brute_force_small():
    rng = np.random.default_rng(21)
    H, I, E, P, T, k = 256, 256, 2, 4, 2, 2
    idx, luts, planes = _make_layer(rng, H, I, E, P, None)
    bits = {(0, 0): 4, (0, 1): 2, (1, 0): 3, (1, 1): 4}
    x = rng.standard_normal((T, H)).astype(np.float16)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    r = apl.route_topk(logits, k)
    y = _oracle_layer(x, r, luts, planes, bits, P, H, I)
    ys = _scalar_layer(x, r["ids"], r["w"], idx, luts, bits, P, H, I, range(T))
    for t in range(T):
        np.testing.assert_allclose(y[t], ys[t], rtol=1e-12, atol=1e-14)


def test_layer_brute_force_tiny_workload_tokens():
    """The tiny workload's shape (H 256, I 512, E 4, top-2, P 4) on a few tokens."""
    from any_precision_bit_pw_gb300 import synth
    wl = synth.TINY_LAYER
    li = synth.layer_inputs(wl)
    H, I, E, P = 256, 512, 4, 4
    idx = {key: v.numpy() for key, v in li.idx.items()}
    luts = {key: {b: t.numpy() for b, t in d.items()} for key, d in li.luts.items()}
    planes = {key: apl.pack_bitplanes(v, P) for key, v in idx.items()}
    bits = {(e, u): li.bits[2 * e + u] for e in range(E) for u in (0, 1)}
    x = li.x.numpy()
    r = apl.route_topk(li.logits.numpy(), 2)
    y = _oracle_layer(x, r, luts, planes, bits, P, H, I)
    toks = [0, 5, 15]
    ys = _scalar_layer(x, r["ids"], r["w"], idx, luts, bits, P, H, I, toks)
    for t in toks:
        np.testing.assert_allclose(y[t], ys[t], rtol=1e-11, atol=1e-13)


def test_layer_reduces_to_dense_ffn():
    """E = 1, k = 1 (so the routing weight is 1): the layer is the dense FFN
    W_dn (silu(W_g x) * (W_u x)) computed by np.matmul on dequantised weights."""
    rng = np.random.default_rng(31)
    H, I, P = 256, 512, 5
    idx, luts, planes = _make_layer(rng, H, I, 1, P, None)
    bits = {(0, 0): 5, (0, 1): 3}
    x = rng.standard_normal((6, H)).astype(np.float16)
    r = apl.route_topk(np.zeros((6, 1), np.float32), 1)
    assert np.all(r["w"] == 1.0)
    y = _oracle_layer(x, r, luts, planes, bits, P, H, I)
    Wgu = np.take_along_axis(luts[0, 0][5].astype(np.float64), idx[0, 0].astype(np.int64) >> 0, axis=1)
    Wdn = np.take_along_axis(luts[0, 1][3].astype(np.float64), idx[0, 1].astype(np.int64) >> 2, axis=1)
    xf = x.astype(np.float64)
    g = np.matmul(xf, Wgu[:I].T)
    up = np.matmul(xf, Wgu[I:].T)
    want = np.matmul((g / (1 + np.exp(-g))) * up, Wdn.T)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Page accounting (§3.1, Eq. 3)
# ---------------------------------------------------------------------------
def test_page_bytes_closed_forms():
    # Mixtral-8x7B gate_up (28672 x 4096), seed 3, at 8 bits:
    # 8 planes * 14,680,064 B + 28672 rows * 2 B * (8+16+32+64+128+256)
    assert apl.page_bytes(28672, 4096, 3, 8) == 117_440_512 + 28_901_376
    # down (4096 x 14336) at 8 bits
    assert apl.page_bytes(4096, 14336, 3, 8) == 58_720_256 + 4_128_768
    # at the seed bitwidth only one LUT is resident
    assert apl.page_bytes(4096, 14336, 3, 3) == 3 * 7_340_032 + 4096 * 8 * 2
    with pytest.raises(ValueError):
        apl.page_bytes(4096, 14336, 3, 2)


def test_eq3_released_bytes_telescope():
    N, K, S = 1024, 512, 3
    total = sum(apl.released_bytes(N, K, S, b, b - 1) for b in range(8, S, -1))
    assert total == apl.released_bytes(N, K, S, 8, S)
    # lowering by one releases one plane and one LUT
    assert apl.released_bytes(N, K, S, 6, 5) == N * K // 8 + N * 64 * 2
    with pytest.raises(ValueError):
        apl.released_bytes(N, K, S, 4, 4)


def test_compare_metrics():
    y = np.array([[3.0, 4.0]])
    m = apl.compare(y, y + np.array([[0.0, 0.05]]))
    assert abs(m["rel_l2"] - 0.01) < 1e-12
    assert abs(m["max_abs"] - 0.05) < 1e-12


def test_index_block_equals_plane_block():
    """The definition path (idx >> (P - q)) and the packed-plane path agree
    exactly, so either may serve as the oracle of a block."""
    rng = np.random.default_rng(41)
    N, K, P = 128, 512, 8
    idx = _rand_idx(rng, N, K, P)
    planes = apl.pack_bitplanes(idx, P)
    luts = {b: np.sort(rng.standard_normal((N, 1 << b)).astype(np.float16), axis=1) for b in range(2, 9)}
    x = rng.standard_normal((3, K)).astype(np.float16)
    for q in (2, 3, 5, 8):
        a = apl.Block(planes, luts, q, N, K).linear(x)
        b = apl.IndexBlock(idx, luts, q, P).linear(x)
        assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# Tiled LUT layout (the library's documented storage of LUT pages)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N,b,n,c,byte", [
    (256, 3, 0, 0, 0),            # strip 0, w 0, i 0, line 0
    (256, 3, 1, 0, 4),            # i 1 -> next word
    (256, 3, 16, 0, 128),         # w 1 -> words 32.. (odd w)
    (256, 3, 32, 0, 2),           # w 2 -> high half-word of word 0
    (256, 3, 48, 5, 5 * 256 + 128 + 2),   # w 3, line 5
    (256, 3, 128, 0, 64),         # second half of the rows: i = 16
    (256, 3, 64, 0, 8 * 256),     # strip 1 starts after 2^b lines
    (256, 4, 64 + 17, 9, (16 + 9) * 256 + 4 * (32 + 1)),
])
def test_lut_layout_hand_derived_points(N, b, n, c, byte):
    assert int(apl.lut_tiled_offset(n, c, N, b)) == byte


@pytest.mark.parametrize("N,b", [(128, 2), (256, 3), (384, 8), (1024, 5)])
def test_lut_layout_is_a_bijection_onto_even_bytes(N, b):
    off = apl.lut_tiled_offset(np.arange(N)[:, None], np.arange(1 << b)[None, :], N, b).ravel()
    assert np.array_equal(np.sort(off), np.arange(0, N * (2 << b), 2))
    # a strip's table is one contiguous run of 2^b * 256 bytes
    strips = (np.arange(N) % (N // 2)) // 64
    for s in range(N // 128):
        rows = np.nonzero(strips == s)[0]
        o = apl.lut_tiled_offset(rows[:, None], np.arange(1 << b)[None, :], N, b)
        assert o.min() == s * (256 << b) and o.max() == (s + 1) * (256 << b) - 2


def test_pack_lut_tiled_places_every_entry():
    rng = np.random.default_rng(5)
    N, b = 256, 4
    lut = rng.standard_normal((N, 1 << b)).astype(np.float16)
    buf = apl.pack_lut_tiled(lut)
    assert buf.size == N * (2 << b)
    for n in (0, 1, 63, 64, 127, 128, 200, 255):
        for c in (0, 7, 15):
            o = int(apl.lut_tiled_offset(n, c, N, b))
            assert buf[o:o + 2].view(np.float16)[0] == lut[n, c]
