"""Planted mistakes: each plants a plausible error in the oracle (on the CPU,
through monkeypatch) and checks that one of the pins fails on it."""
import numpy as np
import pytest

from oracle import apl
import test_oracle_pins as pins


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_lsb_first_plane_order_is_caught(monkeypatch):
    real = apl.unpack_indices

    def lsb_first(planes, b, N, K, rows=None):
        out = real(planes, b, N, K, rows)
        # reverse the bit order of the b-bit index
        rev = np.zeros_like(out)
        for i in range(b):
            rev |= ((out >> i) & 1) << (b - 1 - i)
        return rev
    monkeypatch.setattr(apl, "unpack_indices", lsb_first)
    _fails(pins.test_overlay_invariant_and_round_trip, 128, 512, 8)


def test_wrong_layout_lane_is_caught(monkeypatch):
    real = apl.bit_address

    def swapped(n, j, N, K):   # swap neighbouring 8-column groups of a word
        j = np.asarray(j)
        return real(n, j ^ 8, N, K)
    monkeypatch.setattr(apl, "bit_address", swapped)
    _fails(pins.test_layout_hand_derived_points, 256, 256, 0, 8, 0, 1)


def test_sigmoid_instead_of_silu_is_caught(monkeypatch):
    monkeypatch.setattr(apl, "silu", lambda z: 1.0 / (1.0 + np.exp(-z)))
    _fails(pins.test_layer_reduces_to_dense_ffn)


def test_gate_up_swapped_is_caught(monkeypatch):
    real = apl.moe_layer

    def swapped(x, ids, w, I, blocks, tokens=None):
        class Swap:
            def __init__(self, b):
                self.b = b

            def linear(self, xx):
                G = self.b.linear(xx)
                return np.concatenate([G[:, I:], G[:, :I]], axis=1)

        def blocks2(e, u):
            return Swap(blocks(e, u)) if u == 0 else blocks(e, u)
        return real(x, ids, w, I, blocks2, tokens)
    monkeypatch.setattr(apl, "moe_layer", swapped)
    _fails(pins.test_layer_reduces_to_dense_ffn)


def test_routing_weight_dropped_is_caught(monkeypatch):
    real = apl.moe_layer
    monkeypatch.setattr(apl, "moe_layer",
                        lambda x, ids, w, I, blocks, tokens=None: real(x, ids, np.ones_like(w), I, blocks, tokens))
    _fails(pins.test_layer_brute_force_small)


def test_tie_break_to_higher_index_is_caught(monkeypatch):
    real = apl.route_topk

    def flipped(logits, k):
        lg = np.asarray(logits)[:, ::-1].copy()
        r = real(lg, k)
        E = lg.shape[1]
        r["ids"] = (E - 1 - r["ids"]).astype(np.int32)
        return r
    monkeypatch.setattr(apl, "route_topk", flipped)
    _fails(pins.test_route_matches_brute_force, 16, 4, 2)


def test_missing_lut_term_in_page_bytes_is_caught(monkeypatch):
    monkeypatch.setattr(apl, "page_bytes", lambda N, K, S, b: b * N * K // 8 + N * (1 << b) * 2)
    _fails(pins.test_page_bytes_closed_forms)
