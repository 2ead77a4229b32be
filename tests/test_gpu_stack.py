"""The stack workload on the GPU: page-table commits release exactly the Eq. 3
bytes ("PagedWeight" arXiv text, §3.1), the caching allocator gets them back,
the table's resident bytes follow the host schedule, and layer outputs match
the oracle under the committed bitwidths at every commit phase.  The full
32-layer, 64-step schedule (down to 40 % of the 8-bit footprint) runs with
page release and with offload to host memory (§3.3); a three-layer reduction
checks the allocator side."""
import numpy as np
import pytest
import torch

from oracle import apl

pytestmark = pytest.mark.gpu

pw = pytest.importorskip("any_precision_bit_pw_gb300.pw")
from any_precision_bit_pw_gb300 import synth  # noqa: E402
from any_precision_bit_pw_gb300.stack import StackRun  # noqa: E402
from oracle import parallel as oracle_parallel  # noqa: E402

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    if not os.path.exists(pw.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    pw.lib()
    torch.cuda.set_device(0)


def _check_layer(run, layer, step, y_dev, bits):
    """Every token of one layer (so every expert it routes to) against the
    oracle at the given committed bits {(e, u): q}; the weights are drawn
    again from the workload's seeds, so the oracle never reads the GPU's
    planes."""
    wl = run.wl
    sh = wl.shape
    x, lg = run.inputs(layer, step)
    r = apl.route_topk(lg.cpu().numpy(), sh.top_k)
    toks = list(range(wl.tokens))
    experts = sorted({int(e) for e in r["ids"].ravel()})
    with oracle_parallel.ExpertFiles() as f:
        for e in experts:
            for u in (0, 1):
                q = bits[(e, u)]
                f.add(e, u, synth.parent_indices(wl, layer, e, u, DEV).cpu().numpy(),
                      synth.lut(wl, layer, e, u, q, DEV).cpu().numpy(), q)
        y_ref = oracle_parallel.layer_rows(f, x.cpu().numpy(), r["ids"], r["w"], sh.intermediate, wl.parent_bits,
                                           toks)
    m = apl.compare(y_ref, y_dev[toks])
    assert m["rel_l2"] <= 2e-3 and m["max_abs_over_rms"] <= 1e-2, (layer, step, m)
    return {q for q in bits.values()}


def test_stack_commits_release_pages_and_keep_parity():
    wl = synth.MIXTRAL_8X7B_STACK
    L = 3
    run = StackRun(wl, DEV, layers=L, commit_every=4, n_commits=2, final_fraction=0.55)
    f8 = run.schedule.f8
    assert run.stack.resident_bytes() == f8
    E = wl.shape.experts
    commits = 0
    for step in range(9):
        layer = step % L
        bits = {(e, u): run.stack.committed_bits(run.stack.block_id(layer, e, u))
                for e in range(E) for u in (0, 1)}
        outs = {}
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        plan, released = run.step(on_layer=lambda l, y: outs.__setitem__(l, y.float().cpu().numpy())
                                  if l == layer else None)
        torch.cuda.synchronize()
        assert int(run.call.status.item()) == 0
        if step in (0, 5, 8):
            _check_layer(run, layer, step, outs[layer], bits)
        if plan:
            commits += 1
            want = sum(run.stack.block_bytes_at(run.stack.block_id(*b), o) -
                       run.stack.block_bytes_at(run.stack.block_id(*b), n) for b, o, n in plan)
            assert released == want > 0
            assert before - torch.cuda.memory_allocated() >= released
            assert run.stack.resident_bytes() == run.schedule.resident_bytes()
            for (l, e, u), _, n in plan:
                assert run.stack.committed_bits(run.stack.block_id(l, e, u)) <= n
    assert commits == 2
    assert run.stack.resident_bytes() <= 0.55 * f8


def test_stack_offload_keeps_host_copies_and_parity():
    """The stack driver in offload mode (§3.3) on a three-layer tiny stack:
    lowering copies the released pages to pinned host memory first; once the
    copies finished, every page above its block's committed bitwidth is
    CPU-resident only and its host bytes are the oracle's packed plane (or
    tiled LUT); layer outputs follow the committed bitwidths; reloading every
    lowered block and raising it back restores the 4-bit outputs."""
    wl = synth.TINY_LAYER.with_(name="tiny_stack", tokens=24, bits_mode="fixed", fixed_bits=4,
                                logits_mode="biased", layers=3)
    run = StackRun(wl, DEV, commit_every=2, n_commits=2, final_fraction=0.6, offload=True)
    st = run.stack
    P, S = wl.parent_bits, wl.seed_bits
    for _ in range(4):
        run.step()            # runs the step boundary (commits at steps 2 and 4)
        run.finish_offloads()
    torch.cuda.synchronize()
    assert run.offloaded_bytes > 0
    assert st.resident_bytes() == run.schedule.resident_bytes()
    lowered = []
    for (layer, e, u), q in run.schedule.bits.items():
        b = st.block_id(layer, e, u)
        assert st.committed_bits(b) == q
        if q == P:
            continue
        lowered.append((b, layer, e, u, q))
        idx = synth.parent_indices(wl, layer, e, u, DEV).cpu().numpy()
        ref_planes = apl.pack_bitplanes(idx, P)
        for page in st.pages_between(b, q, P):
            state, d, h = pw.pw_page_state(st.table, b, page)
            assert state == pw.PW_PAGE_CPU and d == 0 and h != 0
            host = st.host[(b, page)].numpy()
            if page < pw.PW_MAX_BITS:
                assert np.array_equal(host, np.ascontiguousarray(ref_planes[page]).view(np.uint8).reshape(-1))
            else:
                lut = synth.lut(wl, layer, e, u, page - pw.PW_MAX_BITS, DEV).cpu().numpy()
                assert np.array_equal(host, apl.pack_lut_tiled(lut))
    assert lowered
    # outputs at the committed bitwidths
    for layer in range(run.L):
        x, lg = run.inputs(layer, 0)
        y = run.call(layer, x, lg).float().cpu().numpy()
        torch.cuda.synchronize()
        bits = {(e, u): st.committed_bits(st.block_id(layer, e, u)) for e in range(wl.shape.experts) for u in (0, 1)}
        _check_layer(run, layer, 0, y, bits)
    # reload every lowered block and raise it back to the parent bitwidth
    for b, *_ in lowered:
        st.reload(b, P, run.copy_stream)
        assert not st.raise_to(b, P)
    run.finish_offloads()
    for b, *_ in lowered:
        assert st.raise_to(b, P)
    st.sync()
    assert st.resident_bytes() == run.schedule.f8
    for layer in range(run.L):
        x, lg = run.inputs(layer, 0)
        y = run.call(layer, x, lg).float().cpu().numpy()
        torch.cuda.synchronize()
        _check_layer(run, layer, 0, y, {(e, u): P for e in range(wl.shape.experts) for u in (0, 1)})


@pytest.mark.slow
@pytest.mark.parametrize("offload", [False, True], ids=["release", "offload"])
def test_stack32_full_schedule_matches_oracle_every_phase(offload):
    """The stack workload as specified: 32 Mixtral-8x7B-shaped layers, 128
    tokens per step, 64 steps, a commit every 8 steps lowering the blocks
    with the least routing mass down to 40 % of the 8-bit footprint.  In each
    of the 8 phases (between two commits) the outputs of rotating layers
    (two per phase with page release, one with offload) are checked token by
    token against the oracle under the bitwidths committed at that step;
    every commit releases exactly the Eq. 3 bytes and the table's resident
    bytes follow the schedule.  With page release every step runs the 32
    layers in one launch; with offload, one launch per layer."""
    wl = synth.MIXTRAL_8X7B_STACK
    L, E = wl.layers, wl.shape.experts
    # page release runs every step's 32 layers in one launch
    # (pw_moe_route_apl_ffn_layers), offload one launch per layer
    run = StackRun(wl, DEV, commit_every=synth.STACK_COMMIT_EVERY,
                   n_commits=synth.STACK_STEPS // synth.STACK_COMMIT_EVERY - 1, offload=offload,
                   batched=not offload)
    st = run.stack
    f8 = run.schedule.f8
    assert st.resident_bytes() == f8
    per_phase = 1 if offload else 2
    checks, commits, seen_bits = 0, 0, set()
    for step in range(synth.STACK_STEPS):
        phase, pos = divmod(step, synth.STACK_COMMIT_EVERY)
        layers = [(3 + 11 * phase + 16 * j) % L for j in range(per_phase)] if pos == 2 else []
        bits = {l: {(e, u): st.committed_bits(st.block_id(l, e, u)) for e in range(E) for u in (0, 1)}
                for l in layers}
        outs = {}
        plan, released = run.step(on_layer=lambda l, y: outs.__setitem__(l, y.float().cpu().numpy())
                                  if l in layers else None)
        torch.cuda.synchronize()
        assert run.status() == 0, step
        for l in layers:
            seen_bits |= _check_layer(run, l, step, outs[l], bits[l])
            checks += 1
        if plan:
            commits += 1
            want = sum(st.block_bytes_at(st.block_id(*b), o) - st.block_bytes_at(st.block_id(*b), n)
                       for b, o, n in plan)
            assert released == want > 0
            assert st.resident_bytes() == run.schedule.resident_bytes()
        if offload:
            run.finish_offloads()
    assert commits == synth.STACK_STEPS // synth.STACK_COMMIT_EVERY - 1
    assert checks == per_phase * synth.STACK_STEPS // synth.STACK_COMMIT_EVERY
    assert st.resident_bytes() <= 0.4 * f8 * 1.001
    assert st.resident_bytes() > 0.3 * f8
    assert min(seen_bits) == wl.seed_bits and max(seen_bits) == wl.parent_bits
    if offload:
        assert run.offloaded_bytes > 0.5 * f8
