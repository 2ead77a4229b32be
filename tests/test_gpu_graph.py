"""GPU: the fused calls inside a CUDA graph.

A caller that captures its decode step into a CUDA graph replays the library's
launches without host work.  Each call below runs once eagerly, is captured
on a side stream, and the graph is replayed twice; the replayed output equals
the eager one bit for bit and the status stays 0.  Covered: the routed call
whose routing runs inside the fused launch (a batch one warp routes), the
routed call with a routing launch before the fused launch (more experts than
one warp routes; the fused kernel is launched with a programmatic
dependency), the unrouted call, and the allocation-free entry point (its
scratch address is looked up by the eager call, before the capture)."""
import os

import pytest
import torch

pytestmark = pytest.mark.gpu

pw = pytest.importorskip("any_precision_bit_pw_gb300.pw")
from any_precision_bit_pw_gb300 import synth  # noqa: E402
from any_precision_bit_pw_gb300.layer import APLMoEStack, MoECall, load_layer  # noqa: E402

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not os.path.exists(pw.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    pw.lib()
    torch.cuda.set_device(0)


def _layer(wl):
    sh = wl.shape
    st = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, wl.parent_bits, wl.seed_bits, DEV,
                     shared=sh.shared)
    li = synth.layer_inputs(wl, device=DEV)
    load_layer(st, 0, li)
    st.sync()
    return st, li


def _eager_then_graph(fn, out, status):
    """Runs fn eagerly on a side stream, captures it, replays the graph twice;
    returns (eager output, replayed output)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return want, out


SHAPES = [
    ("in_kernel_routing", synth.TINY_LAYER.with_(tokens=24)),
    ("routing_launch", synth.TINY_LAYER.with_(tokens=24, shape=synth.MoEShape(256, 512, 12, 2, shared=1))),
]


@pytest.mark.parametrize("name,wl", SHAPES, ids=[s[0] for s in SHAPES])
def test_routed_call_in_a_graph(name, wl):
    st, li = _layer(wl)
    call = MoECall(st, wl.tokens)
    x = li.x.to(DEV).contiguous()
    lg = li.logits.to(DEV).contiguous()
    want, got = _eager_then_graph(lambda: call(0, x, lg, accumulate_mass=False), call.y, call.status)
    assert torch.equal(want, got), name


def test_unrouted_and_noalloc_calls_in_a_graph():
    wl = synth.TINY_LAYER.with_(tokens=24)
    st, li = _layer(wl)
    sh = wl.shape
    call = MoECall(st, wl.tokens)
    x = li.x.to(DEV).contiguous()
    call(0, x, li.logits.to(DEV).contiguous(), accumulate_mass=False)
    torch.cuda.synchronize()
    r = call.route
    K = st.k + st.shared

    def unrouted():
        pw.pw_moe_apl_ffn(st.desc, 0, x, sh.intermediate, st.E, K, r.ids, r.w, r.offsets, r.perm, r.inv_perm,
                          call.ws, call.y, call.status)

    want, got = _eager_then_graph(unrouted, call.y, call.status)
    assert torch.equal(want, got)

    y2 = torch.empty_like(call.y)

    def noalloc():
        pw.pw_moe_apl_ffn_noalloc(st.desc, 0, x, sh.intermediate, st.E, K, r.ids, r.w, r.offsets, r.perm,
                                  r.inv_perm, y2, call.status)

    want2, got2 = _eager_then_graph(noalloc, y2, call.status)
    assert torch.equal(want2, got2)
    assert torch.equal(want2, want)
