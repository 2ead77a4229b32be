"""The allocation-free entry point, pw_moe_apl_ffn_noalloc.

Some callers cannot allocate device memory at call time -- code running under
CUDA graph capture, plugin hosts whose memory contract forbids allocation
during inference, real-time loops that cannot afford an allocation's latency
or failure.  For them libpw runs the fused layer with a fixed scratch array of
its own.  This test calls that entry point through the C ABI twice in a row and
checks each result against the regular entry point (caller workspace): both
run the same kernel with a fixed reduction order, so the outputs must be equal
bit for bit (a scratch layout or aliasing fault that perturbs the output only
slightly still fails); on the tiny layer the output is also checked against
the CPU oracle within the tolerance of the other layer tests.  The file name
sorts last so that a run stopping at the first failure has already run every
other test.
"""
import os

import numpy as np
import pytest
import torch

from oracle import apl

pytestmark = pytest.mark.gpu

pw = pytest.importorskip("any_precision_bit_pw_gb300.pw")
from any_precision_bit_pw_gb300 import synth  # noqa: E402
from any_precision_bit_pw_gb300.layer import APLMoEStack, MoECall, load_layer  # noqa: E402

REL_L2 = 2e-3
MAX_ABS_OVER_RMS = 1e-2
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


def _noalloc(call, stack, x):
    r = call.route
    y = torch.full_like(call.y, float("nan"))
    status = torch.zeros((1,), dtype=torch.int32, device=DEV)
    pw.pw_moe_apl_ffn_noalloc(stack.desc, 0, x, stack.I, stack.E, stack.k, r.ids, r.w, r.offsets, r.perm,
                              r.inv_perm, y, status)
    return y, status


@pytest.mark.parametrize("wl", [synth.TINY_LAYER, synth.MIXTRAL_8X7B_DECODE], ids=lambda w: w.name)
def test_noalloc_matches_workspace_entry_point_twice(wl):
    sh = wl.shape
    dev_inputs = wl.shape.hidden >= 4096
    li = synth.layer_inputs(wl, device=DEV if dev_inputs else "cpu")
    stack = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, wl.parent_bits, wl.seed_bits, DEV)
    load_layer(stack, 0, li)
    stack.sync()
    call = MoECall(stack, wl.tokens)
    for step in range(2):
        x = synth.activations(wl, 0, step, DEV)
        lg = synth.router_logits(wl, 0, step, DEV)
        y_ref = call(0, x, lg).float().cpu().numpy()          # regular entry point, caller workspace
        y, status = _noalloc(call, stack, x)                   # same routing buffers
        torch.cuda.synchronize()
        assert int(call.status.item()) == 0 and int(status.item()) == 0
        y = y[: wl.tokens].float().cpu().numpy()
        assert np.all(np.isfinite(y))
        assert np.array_equal(y_ref, y), (step, apl.compare(y_ref, y))
        if not dev_inputs:
            ids = call.route.ids[: wl.tokens].cpu().numpy()
            r = apl.route_topk(lg.cpu().numpy(), sh.top_k)
            assert np.array_equal(ids, r["ids"])

            def blocks(e, u):
                return apl.IndexBlock(li.idx[(e, u)].numpy(), {b: t.numpy() for b, t in li.luts[(e, u)].items()},
                                      li.bits[2 * e + u], wl.parent_bits)
            y_or = apl.moe_layer(x.cpu().numpy(), r["ids"], r["w"], sh.intermediate, blocks)
            m = apl.compare(y_or, y)
            assert m["rel_l2"] <= REL_L2 and m["max_abs_over_rms"] <= MAX_ABS_OVER_RMS, (step, m)


def test_noalloc_on_the_prefill_path_of_the_8x7b_layer():
    """192 tokens of the 8x7B shape take the prefill path (48 assignments per
    expert), whose workspace fits the array although the decode path's would
    not: the call runs and equals the caller-workspace call bit for bit."""
    wl = synth.MIXTRAL_8X7B_DECODE.with_(tokens=192)
    sh = wl.shape
    li = synth.layer_inputs(wl, device=DEV)
    stack = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, wl.parent_bits, wl.seed_bits, DEV)
    load_layer(stack, 0, li)
    stack.sync()
    call = MoECall(stack, wl.tokens)
    y_ref = call(0, li.x, li.logits).float().cpu().numpy()
    y, status = _noalloc(call, stack, li.x)
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0 and int(status.item()) == 0
    assert np.array_equal(y_ref, y[: wl.tokens].float().cpu().numpy())


def test_noalloc_rejects_calls_beyond_its_scratch():
    # 8x7B shape at 512 tokens needs far more than the 32 MiB array
    assert pw.pw_moe_apl_ffn_workspace(512, 4096, 14336, 8, 2) > pw.PW_NOALLOC_SCRATCH_BYTES
    L = pw.lib()
    rc = L.pw_moe_apl_ffn_noalloc(None, 0, None, 512, 4096, 14336, 8, 2, None, None, None, None, None, None,
                                  None, None)
    assert rc == pw.PW_ERR_WORKSPACE
    assert "scratch" in pw.pw_last_error()
