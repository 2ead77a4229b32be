"""The stack workload on the GPU, reduced to three layers and two commit
points: page-table commits release exactly the Eq. 3 bytes ("PagedWeight"
arXiv text, §3.1), the caching allocator gets them back, the table's resident
bytes follow the host schedule, and layer outputs match the oracle under the
committed bitwidths before and after each commit."""
import numpy as np
import pytest
import torch

from oracle import apl

pytestmark = pytest.mark.gpu

pw = pytest.importorskip("any_precision_bit_pw_gb300.pw")
from any_precision_bit_pw_gb300 import synth  # noqa: E402
from any_precision_bit_pw_gb300.stack import StackRun  # noqa: E402

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
    """Oracle output of two sampled tokens of one layer at the given committed
    bits {(e, u): q}."""
    wl = run.wl
    sh = wl.shape
    x, lg = run.inputs(layer, step)
    r = apl.route_topk(lg.cpu().numpy(), sh.top_k)
    toks = sorted(np.random.default_rng(step * 31 + layer).choice(wl.tokens, 2, replace=False).tolist())
    cache = {}

    def blocks(e, u):
        if (e, u) not in cache:
            q = bits[(e, u)]
            idx = synth.parent_indices(wl, layer, e, u, DEV).cpu().numpy()
            luts = {q: synth.lut(wl, layer, e, u, q, DEV).cpu().numpy()}
            cache[(e, u)] = apl.IndexBlock(idx, luts, q, wl.parent_bits)
        return cache[(e, u)]
    y_ref = apl.moe_layer(x.cpu().numpy(), r["ids"], r["w"], sh.intermediate, blocks, tokens=toks)
    m = apl.compare(y_ref[toks], y_dev[toks])
    assert m["rel_l2"] <= 2e-3 and m["max_abs_over_rms"] <= 1e-2, (layer, step, m)


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
