"""GPU: the routed layer call (routing and the fused expert layer in one
launch, pw_moe_route_apl_ffn) against the two-launch call (pw_moe_route_topk,
then pw_moe_apl_ffn) on the same inputs -- the routing arrays, the routing
mass and y must agree bit for bit -- and against the CPU oracle."""
import numpy as np
import pytest
import torch

from oracle import apl

pytestmark = pytest.mark.gpu

pw = pytest.importorskip("any_precision_bit_pw_gb300.pw")
from any_precision_bit_pw_gb300 import synth  # noqa: E402
from any_precision_bit_pw_gb300.layer import APLMoEStack, MoECall, load_layer  # noqa: E402
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


def _stack(li):
    sh = li.wl.shape
    st = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, li.wl.parent_bits, li.wl.seed_bits, DEV,
                     shared=sh.shared)
    load_layer(st, 0, li)
    st.sync()
    return st


def _oracle_rows(li, tokens):
    """Oracle rows y[tokens] at the committed bitwidths (one expert per host
    core) and the oracle's routing."""
    sh = li.wl.shape
    lg = li.logits.cpu().numpy()
    r = apl.route_topk_shared(lg, sh.top_k, sh.shared) if sh.shared else apl.route_topk(lg, sh.top_k)
    experts = sorted({int(e) for e in r["ids"][tokens].ravel()})
    with oracle_parallel.ExpertFiles() as f:
        for e in experts:
            for u in (0, 1):
                q = li.bits[2 * e + u]
                f.add(e, u, li.idx[(e, u)].cpu().numpy(), li.luts[(e, u)][q].cpu().numpy(), q)
        y = oracle_parallel.layer_rows(f, li.x.cpu().numpy(), r["ids"], r["w"], sh.intermediate,
                                       li.wl.parent_bits, tokens)
    return y, r


def _routing(call):
    r = call.route
    return [t.cpu().numpy().copy() for t in (r.ids, r.w, r.offsets, r.perm, r.inv_perm)]


# (workload, tokens): 16-token tiles, 32-token tiles, the prefill path (a
# routing launch before the fused one), and a tiny shape
CASES = [("tiny", 16), ("tiny", 40), ("8x7b", 32), ("8x7b", 100), ("8x7b", 256), ("8x7b", 3)]


def _inputs(name, T):
    wl = synth.TINY_LAYER if name == "tiny" else synth.MIXTRAL_8X7B_DECODE
    return synth.layer_inputs(wl.with_(tokens=T), device=DEV)


@pytest.mark.parametrize("name,T", CASES)
def test_routed_call_equals_two_launch_call(name, T):
    li = _inputs(name, T)
    st = _stack(li)
    fused, split = MoECall(st, T, fused=True), MoECall(st, T, fused=False)
    for rep in range(3):   # the routing mass accumulates across calls
        yf = fused(0, li.x, li.logits).clone()
        ys = split(0, li.x, li.logits).clone()
        torch.cuda.synchronize()
        assert int(fused.status.item()) == 0 and int(split.status.item()) == 0
        for a, b in zip(_routing(fused), _routing(split)):
            assert np.array_equal(a, b)
        assert torch.equal(yf, ys)
        assert torch.equal(fused.mass, split.mass)
    # and the routing is the oracle's
    r = apl.route_topk(li.logits.cpu().numpy(), li.wl.shape.top_k)
    ids, w, offsets, perm, inv_perm = _routing(fused)
    assert np.array_equal(ids, r["ids"])
    assert np.array_equal(offsets, r["offsets"])
    assert np.array_equal(perm, r["perm"])
    assert np.array_equal(inv_perm, r["inv_perm"])
    np.testing.assert_allclose(w, r["w"], atol=1e-6, rtol=0)


def test_routed_call_matches_oracle_8x7b_decode():
    li = synth.layer_inputs(synth.MIXTRAL_8X7B_DECODE, device=DEV)
    st = _stack(li)
    call = MoECall(st, li.x.shape[0], fused=True)
    y = call(0, li.x, li.logits).float().cpu().numpy()
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0
    toks = list(range(li.x.shape[0]))     # every token
    y_ref, r = _oracle_rows(li, toks)
    assert np.array_equal(call.route.ids.cpu().numpy(), r["ids"])
    m = apl.compare(y_ref, y[toks])
    assert m["rel_l2"] <= 2e-3 and m["max_abs_over_rms"] <= 1e-2, m


def test_routed_call_zero_tokens():
    li = _inputs("tiny", 16)
    st = _stack(li)
    call = MoECall(st, 0, fused=True)
    sh = li.wl.shape
    call.route.offsets.fill_(-1)
    x = torch.empty((0, sh.hidden), dtype=torch.float16, device=DEV)
    lg = torch.empty((0, sh.experts), dtype=torch.float32, device=DEV)
    pw.pw_moe_route_apl_ffn(st.desc, 0, x, lg, sh.intermediate, sh.experts, sh.top_k, call.route.ids,
                            call.route.w, call.route.offsets, call.route.perm, call.route.inv_perm, None, call.ws,
                            call.y, call.status)
    torch.cuda.synchronize()
    assert call.route.offsets.cpu().tolist() == [0] * (sh.experts + 1)


# ---------------------------------------------------------------------------
# shared experts (Table 1: 60 routed + 4 shared top-4; 128 routed + 1 shared top-8)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,E,k,S", [(32, 60, 4, 4), (32, 128, 8, 1), (300, 60, 4, 4), (5, 8, 2, 3)])
def test_route_shared_matches_oracle(T, E, k, S):
    g = torch.Generator().manual_seed(T + E + k + S)
    logits = torch.randn((T, E), generator=g)
    K = k + S
    ids = torch.empty((T, K), dtype=torch.int32, device=DEV)
    w = torch.empty((T, K), dtype=torch.float32, device=DEV)
    off = torch.empty((E + S + 1,), dtype=torch.int32, device=DEV)
    perm = torch.empty((T * K,), dtype=torch.int32, device=DEV)
    inv = torch.empty((T * K,), dtype=torch.int32, device=DEV)
    mass = torch.zeros((E + S,), dtype=torch.float32, device=DEV)
    pw.pw_moe_route_topk_shared(logits.to(DEV).contiguous(), k, S, ids, w, off, perm, inv, mass)
    torch.cuda.synchronize()
    ref = apl.route_topk_shared(logits.numpy(), k, S)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(off.cpu().numpy(), ref["offsets"])
    assert np.array_equal(perm.cpu().numpy(), ref["perm"])
    assert np.array_equal(inv.cpu().numpy(), ref["inv_perm"])
    np.testing.assert_allclose(w.cpu().numpy(), ref["w"], atol=1e-6, rtol=0)
    np.testing.assert_allclose(mass.cpu().numpy() / (T * (1 + S)), ref["mass"], atol=1e-5, rtol=0)


@pytest.mark.parametrize("name", ["qwen15moe_decode_mixed", "gemma4like_decode_mixed"])
def test_shared_expert_layers(name):
    """The Qwen- and Gemma-shaped decode layers: routed call == two-launch call
    bit for bit, and every token against the oracle."""
    wl = synth.WORKLOADS[name]
    li = synth.layer_inputs(wl, device=DEV)
    st = _stack(li)
    sh = wl.shape
    fused, split = MoECall(st, wl.tokens, fused=True), MoECall(st, wl.tokens, fused=False)
    yf = fused(0, li.x, li.logits).clone()
    ys = split(0, li.x, li.logits).clone()
    torch.cuda.synchronize()
    assert int(fused.status.item()) == 0 and int(split.status.item()) == 0
    for a, b in zip(_routing(fused), _routing(split)):
        assert np.array_equal(a, b)
    assert torch.equal(yf, ys)
    toks = list(range(wl.tokens))          # every token, so every routed and shared expert
    y_ref, r = _oracle_rows(li, toks)
    assert np.array_equal(_routing(fused)[0], r["ids"])
    m = apl.compare(y_ref, yf.float().cpu().numpy()[toks])
    assert m["rel_l2"] <= 2e-3 and m["max_abs_over_rms"] <= 1e-2, m


@pytest.mark.parametrize("name,T", [("8x7b", 32), ("8x7b", 100), ("tiny", 40), ("8x7b", 256)])
def test_strip_combine_equals_grid_combine(name, T):
    """The two combine placements (whole grid after the last unit, or each
    strip in the CTA of its last down unit) add the same terms in the same
    order: y is identical bit for bit."""
    li = _inputs(name, T)
    st = _stack(li)
    call = MoECall(st, T)
    y_grid = call(0, li.x, li.logits).clone()
    opts = pw.pw_ffn_options()
    opts.flags = pw.PW_FFN_FLAG_STRIP_COMBINE
    y_strip = call(0, li.x, li.logits, options=opts).clone()
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0
    assert torch.equal(y_grid, y_strip)
