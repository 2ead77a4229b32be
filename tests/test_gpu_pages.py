"""GPU: asynchronous page movement (PagedWeight §3.1 page states, §3.3 and
Figure 4).  Offload copies pages to host memory and lowers q_i at once; the
GPU pages are retired only after the copy finished.  Reload restores pages
first; q_i can be raised only after the copies finished.  The layer output
follows the committed bitwidths throughout (checked against the oracle), the
pages come back byte for byte, and copies on a second stream overlap the
fused layer without changing its output."""
import numpy as np
import pytest
import torch

from oracle import apl

pytestmark = pytest.mark.gpu

pw = pytest.importorskip("any_precision_bit_pw_gb300.pw")
from any_precision_bit_pw_gb300 import synth  # noqa: E402
from any_precision_bit_pw_gb300.layer import APLMoEStack, MoECall, load_layer  # noqa: E402

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


def _layer(bits_all):
    """The tiny layer with every block committed at `bits_all` (its parent)."""
    wl = synth.TINY_LAYER.with_(tokens=24)
    li = synth.layer_inputs(wl, device=DEV)
    li.bits = [bits_all] * len(li.bits)
    sh = wl.shape
    st = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, wl.parent_bits, wl.seed_bits, DEV)
    load_layer(st, 0, li)
    st.sync()
    return li, st


def _oracle(li, bits):
    sh = li.wl.shape
    r = apl.route_topk(li.logits.cpu().numpy(), sh.top_k)

    def blocks(e, u):
        idx = li.idx[(e, u)].cpu().numpy()
        return apl.IndexBlock(idx, {b: t.cpu().numpy() for b, t in li.luts[(e, u)].items()}, bits[2 * e + u],
                              li.wl.parent_bits)
    return apl.moe_layer(li.x.cpu().numpy(), r["ids"], r["w"], sh.intermediate, blocks)


def _check(li, call, bits):
    y = call(0, li.x, li.logits).float().cpu().numpy()
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0
    m = apl.compare(_oracle(li, bits), y)
    assert m["rel_l2"] <= 2e-3 and m["max_abs_over_rms"] <= 1e-2, m
    return y


def _poll_until_done(st, limit_s=10.0):
    import time
    t0 = time.time()
    while st.poll() > 0:
        assert time.time() - t0 < limit_s, "page transfers did not finish"
        time.sleep(0.001)


def test_offload_then_reload_round_trip():
    P = synth.TINY_LAYER.parent_bits
    li, st = _layer(P)
    call = MoECall(st, li.x.shape[0])
    y_full = _check(li, call, [P] * st.n_blocks)
    blk, lo = 3, st.S                      # expert 1's down block, down to the seed bitwidth
    pages = st.pages_between(blk, lo, P)
    originals = {}
    for page in pages:
        t = st.planes[blk][page] if page < pw.PW_MAX_BITS else st.luts[blk][page - pw.PW_MAX_BITS]
        originals[page] = t.view(torch.uint8).reshape(-1).cpu().clone()
    copy = torch.cuda.Stream()
    resident0 = st.resident_bytes()

    # offload: copies start, q_i drops at once, GPU pages stay until the copies finish
    released = st.offload(blk, lo, copy)
    assert st.committed_bits(blk) == lo
    assert released == st.block_bytes_at(blk, P) - st.block_bytes_at(blk, lo)      # Eq. 3
    assert st.resident_bytes() == resident0 - released
    for page in pages:
        state, _, _ = pw.pw_page_state(st.table, blk, page)
        assert state & pw.PW_PAGE_CPU == 0
        if state & pw.PW_PAGE_TO_CPU:
            assert state & pw.PW_PAGE_GPU           # in flight: still attached
    copy.synchronize()
    _poll_until_done(st)
    for page in pages:
        state, d, h = pw.pw_page_state(st.table, blk, page)
        assert state == pw.PW_PAGE_CPU and d == 0 and h != 0
        host = st.host[(blk, page)]
        assert torch.equal(host[: originals[page].numel()], originals[page])
        if page < pw.PW_MAX_BITS:
            assert st.planes[blk][page] is None
        else:
            assert (page - pw.PW_MAX_BITS) not in st.luts[blk]
    st.sync()
    bits = [P] * st.n_blocks
    bits[blk] = lo
    _check(li, call, bits)

    # reload: the copies start, raising is refused until a poll saw them finish
    st.reload(blk, P, copy)
    for page in pages:
        state, _, _ = pw.pw_page_state(st.table, blk, page)
        assert state & pw.PW_PAGE_TO_GPU and not state & pw.PW_PAGE_GPU
    assert not st.raise_to(blk, P)
    assert st.committed_bits(blk) == lo
    copy.synchronize()
    _poll_until_done(st)
    for page in pages:
        state, d, _ = pw.pw_page_state(st.table, blk, page)
        assert state == (pw.PW_PAGE_GPU | pw.PW_PAGE_CPU) and d != 0
        t = st.planes[blk][page] if page < pw.PW_MAX_BITS else st.luts[blk][page - pw.PW_MAX_BITS]
        assert torch.equal(t.view(torch.uint8).reshape(-1)[: originals[page].numel()].cpu(), originals[page])
    assert st.raise_to(blk, P)
    assert st.resident_bytes() == resident0
    st.sync()
    y_back = _check(li, call, [P] * st.n_blocks)
    assert np.array_equal(y_back, y_full)

    # lowering again reuses the host copies: nothing is copied, pages go at once
    released = st.offload(blk, lo, copy)
    assert released == st.block_bytes_at(blk, P) - st.block_bytes_at(blk, lo)
    for page in pages:
        assert pw.pw_page_state(st.table, blk, page)[0] == pw.PW_PAGE_CPU


def test_page_moves_overlap_the_layer():
    """Offload and reload of several blocks on a copy stream while the fused
    layer runs repeatedly on the compute stream: every call's output is the
    one its committed bitwidths give."""
    P = synth.TINY_LAYER.parent_bits
    li, st = _layer(P)
    call = MoECall(st, li.x.shape[0])
    y_full = _check(li, call, [P] * st.n_blocks)
    copy = torch.cuda.Stream()
    moving = [0, 5, 6]
    for b in moving:
        st.offload(b, st.S, copy)
    # the layer keeps running (on the committed, lowered bits) while copies run
    st.sync()
    bits = [P] * st.n_blocks
    for b in moving:
        bits[b] = st.S
    outs = [call(0, li.x, li.logits).clone() for _ in range(5)]
    copy.synchronize()
    _poll_until_done(st)
    torch.cuda.synchronize()
    y_low = _check(li, call, bits)
    for o in outs:
        assert np.array_equal(o.float().cpu().numpy(), y_low)
    for b in moving:
        st.reload(b, P, copy)
    outs = [call(0, li.x, li.logits).clone() for _ in range(5)]   # still the lowered bits
    copy.synchronize()
    _poll_until_done(st)
    for b in moving:
        assert st.raise_to(b, P)
    st.sync()
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(o.float().cpu().numpy(), y_low)
    assert np.array_equal(_check(li, call, [P] * st.n_blocks), y_full)


def test_transfer_in_flight_is_busy():
    P = synth.TINY_LAYER.parent_bits
    li, st = _layer(P)
    copy = torch.cuda.Stream()
    page = P - 1
    host = torch.empty(pw.pw_page_bytes(st.table, 0, page), dtype=torch.uint8, pin_memory=True)
    # hold the copy stream so the offload cannot finish before the second call
    gate = torch.cuda.Event()
    spin = torch.cuda.Stream()
    with torch.cuda.stream(spin):
        torch.cuda._sleep(20_000_000)
        gate.record(spin)
    copy.wait_event(gate)
    pw.pw_page_offload(st.table, 0, page, host, stream=copy)
    with pytest.raises(pw.PwError) as e:
        pw.pw_page_offload(st.table, 0, page, host, stream=copy)
    assert e.value.code == pw.PW_ERR_BUSY
    with pytest.raises(pw.PwError) as e:
        pw.pw_page_table_attach_plane(st.table, 0, page, st.planes[0][page].data_ptr())
    assert e.value.code == pw.PW_ERR_BUSY
    assert st.poll() >= 1
    torch.cuda.synchronize()
    _poll_until_done(st)
    assert pw.pw_page_state(st.table, 0, page)[0] == pw.PW_PAGE_GPU | pw.PW_PAGE_CPU
