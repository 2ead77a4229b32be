"""GPU: several independent MoE layers in one launch
(pw_moe_route_apl_ffn_layers) against one routed call per layer
(pw_moe_route_apl_ffn) on the same inputs -- outputs, routing arrays (after
the documented index shift) and routing mass agree bit for bit -- and a layer
of the batch against the CPU oracle.  "PagedWeight" arXiv text, §3.3: the
fused kernel runs routing, the experts' projections and the weighted sum of
their outputs; here one persistent launch does so for a stack of layers."""
import numpy as np
import pytest
import torch

from oracle import apl

pytestmark = pytest.mark.gpu

pw = pytest.importorskip("any_precision_bit_pw_gb300.pw")
from any_precision_bit_pw_gb300 import synth  # noqa: E402
from any_precision_bit_pw_gb300.layer import APLMoEStack, MoECall, MoELayersCall, load_layer  # noqa: E402

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


def _stack(wl, L, device_inputs):
    sh = wl.shape
    st = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, L, wl.parent_bits, wl.seed_bits, DEV,
                     shared=sh.shared)
    lis = []
    for layer in range(L):
        li = synth.layer_inputs(wl, layer=layer, device=DEV if device_inputs else "cpu")
        load_layer(st, layer, li)
        lis.append(li)
    st.sync()
    return st, lis


CASES = [
    ("tiny_t16", synth.TINY_LAYER, 3, False),                                  # 16-token tiles, decode path
    ("tiny_prefill", synth.TINY_LAYER.with_(tokens=100), 2, False),            # routing launch first
    ("tiny_shared", synth.TINY_LAYER.with_(tokens=20, shape=synth.MoEShape(256, 512, 4, 2, shared=2)), 3, False),
    ("8x7b_t64", synth.MIXTRAL_8X7B_STACK, 3, True),                           # the stack shape, 64-token tiles
    ("8x7b_t16", synth.MIXTRAL_8X7B_STACK.with_(tokens=8), 4, True),
]


@pytest.mark.parametrize("name,wl,L,dev_inputs", CASES, ids=[c[0] for c in CASES])
def test_layers_call_equals_per_layer_calls(name, wl, L, dev_inputs):
    st, lis = _stack(wl, L, dev_inputs)
    sh = wl.shape
    T, K, ET = wl.tokens, sh.top_k + sh.shared, sh.total_experts
    x = torch.stack([li.x.to(DEV) for li in lis]).contiguous()
    lg = torch.stack([li.logits.to(DEV) for li in lis]).contiguous()
    batched = MoELayersCall(st, T, L)
    single = MoECall(st, T)
    mass_b = torch.zeros((L, ET), dtype=torch.float32, device=DEV)
    for rep in range(2):
        yb = batched(0, x, lg, mass=mass_b).clone()
        torch.cuda.synchronize()
        assert int(batched.status.item()) == 0
        off_b = batched.offsets.cpu().numpy()
        perm_b = batched.perm.cpu().numpy()
        inv_b = batched.inv_perm.cpu().numpy()
        A = T * K
        for layer in range(L):
            ys = single(layer, x[layer], lg[layer]).clone()
            torch.cuda.synchronize()
            assert int(single.status.item()) == 0
            assert torch.equal(yb[layer, :T], ys), (rep, layer)
            r = single.route
            assert torch.equal(batched.ids[layer, :T], r.ids[:T])
            assert torch.equal(batched.w[layer, :T], r.w[:T])
            assert np.array_equal(off_b[layer * ET:(layer + 1) * ET + 1], r.offsets.cpu().numpy() + layer * A)
            assert np.array_equal(perm_b[layer * A:(layer + 1) * A], r.perm.cpu().numpy()[:A] + layer * A)
            assert np.array_equal(inv_b[layer * A:(layer + 1) * A], r.inv_perm.cpu().numpy()[:A] + layer * A)
    assert torch.equal(mass_b, single.mass[:L])     # both accumulated twice, in the same order


def test_layers_call_matches_oracle_tiny():
    wl = synth.TINY_LAYER.with_(tokens=24)
    L = 3
    st, lis = _stack(wl, L, False)
    sh = wl.shape
    call = MoELayersCall(st, wl.tokens, L)
    y = call(0, torch.stack([li.x for li in lis]).to(DEV), torch.stack([li.logits for li in lis]).to(DEV))
    y = y.float().cpu().numpy()
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0
    for layer, li in enumerate(lis):
        r = apl.route_topk(li.logits.numpy(), sh.top_k)
        assert np.array_equal(call.ids[layer].cpu().numpy(), r["ids"])

        def blocks(e, u, li=li):
            N, K = sh.block_shape(u)
            return apl.Block(apl.pack_bitplanes(li.idx[(e, u)].numpy(), wl.parent_bits),
                             {b: t.numpy() for b, t in li.luts[(e, u)].items()}, li.bits[2 * e + u], N, K)
        y_ref = apl.moe_layer(li.x.numpy(), r["ids"], r["w"], sh.intermediate, blocks)
        m = apl.compare(y_ref, y[layer])
        assert m["rel_l2"] <= 2e-3 and m["max_abs_over_rms"] <= 1e-2, (layer, m)


def test_layers_call_starting_at_a_later_layer():
    """layer0 > 0: the call reads the descriptors of layers layer0 .. layer0+L-1."""
    wl = synth.TINY_LAYER
    st, lis = _stack(wl, 4, False)
    x = torch.stack([li.x for li in lis[1:3]]).to(DEV)
    lg = torch.stack([li.logits for li in lis[1:3]]).to(DEV)
    call = MoELayersCall(st, wl.tokens, 2)
    yb = call(1, x, lg).clone()
    single = MoECall(st, wl.tokens)
    for j in range(2):
        ys = single(1 + j, x[j], lg[j])
        torch.cuda.synchronize()
        assert torch.equal(yb[j], ys)
