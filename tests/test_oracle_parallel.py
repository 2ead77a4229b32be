"""The per-expert parallel driver of the oracle (oracle/parallel.py) used by
the full-size GPU parity tests and the CPU baseline: its layer rows equal the
oracle's own moe_layer on the whole layer (the experts' contributions are only
summed in another order), including shared experts and a token subset; its
timing workers run and answer."""
import numpy as np

from any_precision_bit_pw_gb300 import synth
from oracle import apl

from oracle import parallel as oracle_parallel


def _files(li, experts):
    f = oracle_parallel.ExpertFiles()
    for e in experts:
        for u in (0, 1):
            q = li.bits[2 * e + u]
            f.add(e, u, li.idx[(e, u)].numpy(), li.luts[(e, u)][q].numpy(), q)
    return f


def _blocks(li):
    def blocks(e, u):
        return apl.IndexBlock(li.idx[(e, u)].numpy(), {b: t.numpy() for b, t in li.luts[(e, u)].items()},
                              li.bits[2 * e + u], li.wl.parent_bits)
    return blocks


def test_parallel_rows_equal_moe_layer_tiny():
    wl = synth.TINY_LAYER.with_(tokens=24)
    li = synth.layer_inputs(wl)
    sh = wl.shape
    r = apl.route_topk(li.logits.numpy(), sh.top_k)
    want = apl.moe_layer(li.x.numpy(), r["ids"], r["w"], sh.intermediate, _blocks(li))
    toks = list(range(wl.tokens))
    with _files(li, range(sh.experts)) as f:
        got = oracle_parallel.layer_rows(f, li.x.numpy(), r["ids"], r["w"], sh.intermediate, wl.parent_bits, toks,
                                         workers=2)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)


def test_parallel_rows_token_subset_and_shared_experts():
    wl = synth.TINY_LAYER.with_(tokens=20, shape=synth.MoEShape(256, 512, 4, 2, shared=2),
                                bits_choices=(2, 3, 4))
    li = synth.layer_inputs(wl)
    sh = wl.shape
    r = apl.route_topk_shared(li.logits.numpy(), sh.top_k, sh.shared)
    toks = [3, 7, 8, 19]
    want = apl.moe_layer(li.x.numpy(), r["ids"], r["w"], sh.intermediate, _blocks(li), tokens=toks)[toks]
    with _files(li, range(sh.total_experts)) as f:
        got = oracle_parallel.layer_rows(f, li.x.numpy(), r["ids"], r["w"], sh.intermediate, wl.parent_bits, toks,
                                         workers=1)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)


def test_covering_tokens_cover_every_expert_slot_pair():
    rng = np.random.default_rng(3)
    ids = np.stack([rng.permutation(8)[:2] for _ in range(500)]).astype(np.int32)
    toks = oracle_parallel.covering_tokens(ids, extra=5, seed=1)
    pairs = {(int(ids[t, j]), j) for t in range(500) for j in range(2)}
    assert {(int(ids[t, j]), j) for t in toks for j in range(2)} == pairs
    assert len(toks) == len(set(toks)) and len(toks) <= len(pairs) + 5


def test_timing_workers_run_the_layer():
    wl = synth.TINY_LAYER
    li = synth.layer_inputs(wl)
    sh = wl.shape
    r = apl.route_topk(li.logits.numpy(), sh.top_k)
    with _files(li, range(sh.experts)) as f:
        with oracle_parallel.ExpertWorkers(f, li.x.numpy(), r["ids"], r["w"], sh.intermediate,
                                           wl.parent_bits) as ew:
            assert ew.experts == sorted(set(r["ids"].ravel().tolist()))
            assert ew.step(1.0) > 0 and ew.step(0.5) > 0
