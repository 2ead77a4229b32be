"""Host logic of the stack workload's commit schedule (no GPU)."""
import pytest

from oracle import apl
from any_precision_bit_pw_gb300 import stack
from any_precision_bit_pw_gb300.stack import DOWN, GATE_UP

H, I, S, P = 4096, 14336, 3, 8


def _bytes(b, q):
    _, _, u = b
    N, K = (2 * I, H) if u == GATE_UP else (H, I)
    return apl.page_bytes(N, K, S, q)


def test_f8_matches_eq3_sizes():
    sch = stack.StackSchedule(32, 8, S, P, _bytes)
    # 32 layers x 8 experts x (gate_up + down) at 8 bits ~ 53.5 GB
    assert sch.f8 == 32 * 8 * (apl.page_bytes(2 * I, H, S, 8) + apl.page_bytes(H, I, S, 8))
    assert abs(sch.f8 / 1e9 - 53.55) < 0.1


def test_schedule_hits_each_target_and_ends_near_40_percent():
    L, E = 32, 8
    sch = stack.StackSchedule(L, E, S, P, _bytes)
    mass = [[(l * 7 + e * 13) % 11 + 0.5 for e in range(E)] for l in range(L)]
    for step in range(1, 65):
        plan = sch.at_boundary(step, mass)
        if step % 8 or step > 56:
            assert plan == []
            continue
        j = step // 8
        target = stack.byte_target(step, 8, 7, sch.f8)
        assert sch.resident_bytes() <= target
        # minimal: undoing the last lowering step would exceed the target
        b, old, new = plan[-1]
        assert sch.resident_bytes() + _bytes(b, old) - _bytes(b, new) > target
    assert abs(sch.resident_bytes() / sch.f8 - 0.4) < 0.01
    assert min(sch.bits.values()) >= S


def test_lowest_mass_blocks_go_first_down_before_gate_up():
    E = 4
    sch = stack.StackSchedule(1, E, S, P, _bytes)
    mass = [[5.0, 1.0, 3.0, 1.0]]       # experts 1 and 3 tie; expert 1 (lower index) first
    target = sch.f8 - 1                   # one step is enough
    plan = stack.plan_lowering(sch.bits, {(0, e): mass[0][e] for e in range(E)}, _bytes, S, target)
    assert plan == [((0, 1, DOWN), 8, 7)]
    # a deeper target lowers expert 1's down block to the floor, then its gate_up
    dn = _bytes((0, 1, DOWN), 8) - _bytes((0, 1, DOWN), S)
    plan = stack.plan_lowering(sch.bits, {(0, e): mass[0][e] for e in range(E)}, _bytes, S, sch.f8 - dn - 1)
    assert [p[0] for p in plan[:5]] == [(0, 1, DOWN)] * 5
    assert plan[5][0] == (0, 1, GATE_UP)


def test_floor_is_the_seed_bitwidth():
    sch = stack.StackSchedule(2, 2, S, P, _bytes)
    plan = stack.plan_lowering(sch.bits, {}, _bytes, S, 0)
    q = dict(sch.bits)
    for b, old, new in plan:
        assert new == old - 1
        q[b] = new
    assert all(v == S for v in q.values())
    floor = sum(_bytes(b, S) for b in q)
    assert 0.31 < floor / sch.f8 < 0.33   # the q = 3 floor is ~31.8 % of F8
