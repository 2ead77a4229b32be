"""Pins of the oracle's routing with shared experts (the pages' Table 1:
models with routed plus shared experts).  Shared experts take every token
with weight 1; the pins check that reading against structure, the routed-only
routing, and a dense-FFN decomposition of the layer computed with np.matmul."""
import numpy as np
import pytest

from oracle import apl


@pytest.mark.parametrize("T,E,k,S", [(5, 6, 2, 2), (16, 60, 4, 4), (9, 128, 8, 1), (1, 3, 1, 2)])
def test_shared_routing_structure(T, E, k, S):
    rng = np.random.default_rng(T * 1000 + E * 10 + k + S)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    r0 = apl.route_topk(logits, k)
    r = apl.route_topk_shared(logits, k, S)
    K = k + S
    # routed slots are route_topk's, shared slots are experts E..E+S-1 with weight 1
    assert r["ids"].shape == (T, K) and r["w"].shape == (T, K)
    assert np.array_equal(r["ids"][:, :k], r0["ids"])
    np.testing.assert_array_equal(r["w"][:, :k], r0["w"])
    assert np.array_equal(r["ids"][:, k:], np.tile(np.arange(E, E + S), (T, 1)))
    assert np.all(r["w"][:, k:] == 1.0)
    # every shared expert sees every token; the routed experts' counts are route_topk's
    counts = np.diff(r["offsets"])
    assert np.array_equal(counts[:E], np.diff(r0["offsets"]))
    assert np.all(counts[E:] == T)
    # the permutation lists slots by (expert, token, slot): check the keys by brute force
    keys = [(int(r["ids"][s // K, s % K]), s // K, s % K) for s in r["perm"]]
    assert keys == sorted(keys)
    assert sorted(r["perm"].tolist()) == list(range(T * K))
    for pos, s in enumerate(r["perm"]):
        assert r["inv_perm"][s] == pos
    # Eq. 1 over all experts: shared experts get T * 1 of the T * (1 + S) total weight
    np.testing.assert_allclose(r["mass"].sum(), 1.0, rtol=1e-12)
    np.testing.assert_allclose(r["mass"][E:], 1.0 / (1 + S), rtol=1e-12)


def test_shared_routing_without_shared_experts_is_route_topk():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((11, 7)).astype(np.float32)
    a, b = apl.route_topk(logits, 3), apl.route_topk_shared(logits, 3, 0)
    for key in ("ids", "offsets", "perm", "inv_perm"):
        assert np.array_equal(a[key], b[key])
    np.testing.assert_array_equal(a["w"], b["w"])
    np.testing.assert_allclose(a["mass"], b["mass"], rtol=1e-12)


def _dense_ffn(x, idx_gu, lut_gu, idx_dn, lut_dn, P, bg, bd, I):
    Wgu = np.take_along_axis(lut_gu[bg].astype(np.float64), idx_gu.astype(np.int64) >> (P - bg), axis=1)
    Wdn = np.take_along_axis(lut_dn[bd].astype(np.float64), idx_dn.astype(np.int64) >> (P - bd), axis=1)
    xf = x.astype(np.float64)
    g = np.matmul(xf, Wgu[:I].T)
    up = np.matmul(xf, Wgu[I:].T)
    return np.matmul((g / (1 + np.exp(-g))) * up, Wdn.T)


def test_layer_with_shared_experts_is_routed_layer_plus_dense_ffns():
    """y(shared routing) = y(routed-only routing) + sum over shared experts of
    their dense FFN on every token (weight 1)."""
    rng = np.random.default_rng(41)
    H, I, E, S, k, P, T = 128, 128, 4, 2, 2, 4, 7
    idx, luts, bits = {}, {}, {}
    for e in range(E + S):
        for u, (N, K) in ((0, (2 * I, H)), (1, (H, I))):
            idx[e, u] = rng.integers(0, 1 << P, size=(N, K), dtype=np.uint8)
            luts[e, u] = {b: np.sort((rng.standard_normal((N, 1 << b)) * 0.02).astype(np.float16), axis=1)
                          for b in range(1, P + 1)}
            bits[e, u] = int(rng.integers(2, P + 1))
    x = rng.standard_normal((T, H)).astype(np.float16)
    logits = rng.standard_normal((T, E)).astype(np.float32)

    def blocks(e, u):
        return apl.IndexBlock(idx[e, u], luts[e, u], bits[e, u], P)
    rs = apl.route_topk_shared(logits, k, S)
    r0 = apl.route_topk(logits, k)
    y = apl.moe_layer(x, rs["ids"], rs["w"], I, blocks)
    want = apl.moe_layer(x, r0["ids"], r0["w"], I, blocks)
    for s in range(S):
        e = E + s
        want = want + _dense_ffn(x, idx[e, 0], luts[e, 0], idx[e, 1], luts[e, 1], P, bits[e, 0], bits[e, 1], I)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-14)
