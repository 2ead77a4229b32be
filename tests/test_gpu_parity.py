"""GPU parity: libpw's kernels (called through the C ABI) against the CPU
oracle on the same seeded inputs.  Bit-exact for packing, indices, routing ids
and the permutation; rel-L2 <= 2e-3 and max-abs <= 1e-2 * rms(y) for the fp16
layer output (fp32 accumulation), as the fused-kernel target states."""
import numpy as np
import pytest
import torch

from oracle import apl

pytestmark = pytest.mark.gpu

pw = pytest.importorskip("any_precision_bit_pw_gb300.pw")
from any_precision_bit_pw_gb300 import synth  # noqa: E402
from any_precision_bit_pw_gb300.layer import APLMoEStack, MoECall, load_layer  # noqa: E402
from oracle import parallel as oracle_parallel  # noqa: E402

REL_L2 = 2e-3
MAX_ABS_OVER_RMS = 1e-2


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


DEV = "cuda"


def _planes_bytes(planes):
    return [p.view(torch.uint8).cpu().numpy() for p in planes]


# ---------------------------------------------------------------------------
# packer / unpack
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N,K,P", [(128, 128, 1), (128, 256, 8), (256, 512, 8), (1024, 256, 4), (384, 768, 3),
                                   (2048, 4096, 8)])
def test_pack_bytes_match_oracle(N, K, P):
    g = torch.Generator().manual_seed(N + K + P)
    idx = torch.randint(0, 1 << P, (N, K), generator=g, dtype=torch.uint8)
    planes = [torch.empty(N * K // 32, dtype=torch.int32, device=DEV) for _ in range(P)]
    pw.pw_pack_bitplanes(idx.to(DEV), P, planes)
    torch.cuda.synchronize()
    want = apl.pack_bitplanes(idx.numpy(), P)
    for got, ref in zip(_planes_bytes(planes), want):
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("N,b", [(128, 2), (256, 3), (1024, 5), (4096, 8), (28672, 4)])
def test_pack_lut_matches_oracle(N, b):
    g = torch.Generator().manual_seed(N + b)
    lut = (torch.randn((N, 1 << b), generator=g) * 0.02).to(torch.float16)
    out = torch.empty((N, 1 << b), dtype=torch.float16, device=DEV)
    pw.pw_pack_lut(lut.to(DEV).contiguous(), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.view(torch.uint8).cpu().numpy().reshape(-1), apl.pack_lut_tiled(lut.numpy()))


def _table_for(idx_dev, P, S, luts=None, q=None):
    N, K = idx_dev.shape
    t = pw.pw_page_table_create([pw.pw_block_info(N, K, P, S, pw.PW_LAYOUT_TILED, 0)])
    planes = [torch.empty(N * K // 32, dtype=torch.int32, device=DEV) for _ in range(P)]
    pw.pw_pack_bitplanes(idx_dev, P, planes)
    for p in range(P):
        pw.pw_page_table_attach_plane(t, 0, p, planes[p].data_ptr())
    keep = [planes]
    if luts is not None:
        for b, l in luts.items():
            lt = torch.empty_like(l)
            pw.pw_pack_lut(l, lt)           # LUT pages are stored in the tiled LUT layout
            pw.pw_page_table_attach_lut(t, 0, b, lt.data_ptr())
            keep.append(lt)
        pw.pw_page_table_set_bits(t, 0, q)
    return t, keep


@pytest.mark.parametrize("N,K", [(128, 512), (1024, 768)])
def test_unpack_is_top_bits(N, K):
    g = torch.Generator().manual_seed(3)
    idx = torch.randint(0, 256, (N, K), generator=g, dtype=torch.uint8)
    t, keep = _table_for(idx.to(DEV), 8, 3)
    try:
        out = torch.empty((N, K), dtype=torch.uint8, device=DEV)
        for b in range(1, 9):
            pw.pw_unpack_indices(t, 0, b, out)
            torch.cuda.synchronize()
            assert torch.equal(out.cpu(), idx >> (8 - b)), b
    finally:
        pw.pw_page_table_destroy(t)


# ---------------------------------------------------------------------------
# any-precision linear
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("q", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K,M", [(128, 512, 1), (384, 768, 7), (128, 256, 64), (256, 1024, 70), (128, 128, 300)])
def test_apl_linear_matches_oracle(q, N, K, M):
    g = torch.Generator().manual_seed(q * 100 + N + K + M)
    idx = torch.randint(0, 256, (N, K), generator=g, dtype=torch.uint8)
    luts = {b: torch.sort((torch.randn((N, 1 << b), generator=g) * 0.02).half(), dim=1).values
            for b in range(2, 9)}
    x = torch.randn((M, K), generator=g).half()
    t, keep = _table_for(idx.to(DEV), 8, 2, {b: l.to(DEV) for b, l in luts.items() if b <= q}, q)
    try:
        out = torch.empty((M, N), dtype=torch.float32, device=DEV)
        pw.pw_apl_linear(t, 0, x.to(DEV), out)
        torch.cuda.synchronize()
        ref = apl.IndexBlock(idx.numpy(), {b: l.numpy() for b, l in luts.items()}, q, 8).linear(x.numpy())
        m = apl.compare(ref, out.cpu().numpy())
        assert m["rel_l2"] < 1e-5, m
    finally:
        pw.pw_page_table_destroy(t)


@pytest.mark.parametrize("q,N,K,M", [(8, 128, 512, 5), (3, 256, 768, 40), (5, 128, 4096, 3), (2, 128, 128, 17),
                                     (6, 256, 512, 2), (4, 128, 384, 1), (8, 384, 1024, 200)])
def test_apl_linear_identity_lut_is_exact(q, N, K, M):
    """LUT_q[n][c] = c and integer x: the GPU result equals the integer matmul
    of the q-bit indices exactly (every partial sum is an integer < 2^24)."""
    g = torch.Generator().manual_seed(7 + q)
    idx = torch.randint(0, 256, (N, K), generator=g, dtype=torch.uint8)
    lut = torch.arange(1 << q, dtype=torch.float16).repeat(N, 1)
    x = torch.randint(-2, 3, (M, K), generator=g).half()
    luts = {b: (lut if b == q else torch.zeros((N, 1 << b), dtype=torch.float16)).to(DEV) for b in range(2, q + 1)}
    t, keep = _table_for(idx.to(DEV), 8, 2, luts, q)
    try:
        out = torch.empty((M, N), dtype=torch.float32, device=DEV)
        pw.pw_apl_linear(t, 0, x.to(DEV), out)
        torch.cuda.synchronize()
        want = x.long() @ (idx.long() >> (8 - q)).T
        assert torch.equal(out.cpu().double(), want.double())
    finally:
        pw.pw_page_table_destroy(t)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------
def _route_gpu(logits, k):
    T, E = logits.shape
    ids = torch.empty((max(T, 1), k), dtype=torch.int32, device=DEV)
    w = torch.empty((max(T, 1), k), dtype=torch.float32, device=DEV)
    off = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    perm = torch.empty((max(T * k, 1),), dtype=torch.int32, device=DEV)
    inv = torch.empty((max(T * k, 1),), dtype=torch.int32, device=DEV)
    mass = torch.zeros((E,), dtype=torch.float32, device=DEV)
    pw.pw_moe_route_topk(logits.to(DEV).contiguous(), k, ids, w, off, perm, inv, mass)
    torch.cuda.synchronize()
    return dict(ids=ids[:T].cpu().numpy(), w=w[:T].cpu().numpy(), offsets=off.cpu().numpy(),
                perm=perm[:T * k].cpu().numpy(), inv_perm=inv[:T * k].cpu().numpy(), mass=mass.cpu().numpy())


@pytest.mark.parametrize("T,E,k,kind", [(16, 4, 2, "normal"), (32, 8, 2, "normal"), (1, 8, 2, "normal"),
                                        (32, 8, 4, "normal"), (7, 3, 3, "normal"), (32, 4, 2, "ties"),
                                        (31, 8, 2, "ties"), (33, 8, 2, "normal"),
                                        (4096, 8, 2, "zipf"), (2500, 8, 2, "ties"), (3000, 64, 4, "normal"),
                                        (256, 8, 2, "uniform"), (5, 256, 8, "normal"),
                                        (100, 60, 4, "ties"), (40, 128, 8, "ties"), (33, 255, 16, "ties"),
                                        (2000, 33, 3, "ties"), (64, 40, 1, "normal")])
def test_route_matches_oracle(T, E, k, kind):
    g = torch.Generator().manual_seed(T + E + k)
    if kind == "zipf":
        logits = synth.router_logits(synth.MIXTRAL_8X22B_PREFILL, tokens=T)
    elif kind == "uniform":
        logits = synth.router_logits(synth.MIXTRAL_8X7B_SWEEP, tokens=T)
    else:
        logits = torch.randn((T, E), generator=g)
        if kind == "ties":   # many exact ties: quantise the logits
            logits = torch.round(logits * 2) / 2
    got = _route_gpu(logits, k)
    ref = apl.route_topk(logits.numpy(), k)
    assert np.array_equal(got["ids"], ref["ids"])
    assert np.array_equal(got["offsets"], ref["offsets"])
    assert np.array_equal(got["perm"], ref["perm"])
    assert np.array_equal(got["inv_perm"], ref["inv_perm"])
    np.testing.assert_allclose(got["w"], ref["w"], atol=1e-6, rtol=0)
    np.testing.assert_allclose(got["mass"] / max(T, 1), ref["mass"], atol=1e-5, rtol=0)


def test_route_small_batches_many_seeds():
    """Batches of up to 32 tokens over up to 8 experts are routed by one warp
    (ballots instead of a CTA-wide counting sort): every output against the
    oracle over many seeds, tied logits included."""
    for seed in range(40):
        g = torch.Generator().manual_seed(1000 + seed)
        T = 1 + seed % 32
        E = 2 + seed % 7
        k = 1 + seed % min(E, 4)
        logits = torch.randn((T, E), generator=g)
        if seed % 2:
            logits = torch.round(logits * 2) / 2
        got = _route_gpu(logits, k)
        ref = apl.route_topk(logits.numpy(), k)
        for key in ("ids", "offsets", "perm", "inv_perm"):
            assert np.array_equal(got[key], ref[key]), (seed, key)
        np.testing.assert_allclose(got["w"], ref["w"], atol=1e-6, rtol=0)


def test_ffn_rejects_routing_arrays_that_are_not_a_permutation():
    """The unrouted call takes the routing arrays from the caller: an entry
    outside the assignment slots, or offsets that do not run from 0 to T*k,
    set PW_ERR_INVALID_ARG (the kernel's own checks skip the bad entries) and
    the context stays usable."""
    li = synth.layer_inputs(synth.TINY_LAYER)
    sh = li.wl.shape
    y, status, call, stack = _run_gpu(li)
    assert status == 0
    r = call.route
    A = li.wl.tokens * sh.top_k
    for what in ("perm", "inv_perm", "offsets"):
        perm, inv, off = r.perm.clone(), r.inv_perm.clone(), r.offsets.clone()
        if what == "perm":
            perm[3] = A + 7
        elif what == "inv_perm":
            inv[5] = -2
        else:
            off[-1] = A + 16
        call.status.zero_()
        pw.pw_moe_apl_ffn(stack.desc, 0, li.x.to(DEV), sh.intermediate, sh.experts, sh.top_k, r.ids, r.w, off, perm,
                          inv, call.ws, call.y, call.status)
        torch.cuda.synchronize()
        assert int(call.status.item()) == pw.PW_ERR_INVALID_ARG, what
    call.status.zero_()
    y2 = call(0, li.x.to(DEV), li.logits.to(DEV)).float().cpu().numpy()
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0 and np.array_equal(y, y2)


def test_route_zero_tokens():
    got = _route_gpu(torch.zeros((0, 8)), 2)
    assert np.array_equal(got["offsets"], np.zeros(9, np.int32))


# ---------------------------------------------------------------------------
# the fused layer
# ---------------------------------------------------------------------------
def _oracle_y(li, tokens=None, from_planes=False):
    sh, P = li.wl.shape, li.wl.parent_bits
    r = apl.route_topk(li.logits.cpu().numpy(), sh.top_k)
    cache = {}

    def blocks(e, u):
        if (e, u) not in cache:
            idx = li.idx[(e, u)].cpu().numpy()
            luts = {b: t.cpu().numpy() for b, t in li.luts[(e, u)].items()}
            q = li.bits[2 * e + u]
            if from_planes:
                N, K = idx.shape
                cache[(e, u)] = apl.Block(apl.pack_bitplanes(idx, P), luts, q, N, K)
            else:
                cache[(e, u)] = apl.IndexBlock(idx, luts, q, P)
        return cache[(e, u)]
    return apl.moe_layer(li.x.cpu().numpy(), r["ids"], r["w"], sh.intermediate, blocks, tokens=tokens), r


def _run_gpu(li, options=None):
    sh = li.wl.shape
    stack = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, li.wl.parent_bits,
                        li.wl.seed_bits, DEV)
    load_layer(stack, 0, li)
    stack.sync()
    call = MoECall(stack, li.x.shape[0])
    y = call(0, li.x.to(DEV), li.logits.to(DEV), options=options)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), int(call.status.item()), call, stack


def _assert_close(y_ref, y, rows=None):
    if rows is not None:
        y_ref, y = y_ref[rows], y[rows]
    m = apl.compare(y_ref, y)
    assert m["rel_l2"] <= REL_L2 and m["max_abs_over_rms"] <= MAX_ABS_OVER_RMS, m
    return m


def test_ffn_tiny_workload():
    li = synth.layer_inputs(synth.TINY_LAYER)
    y, status, call, _ = _run_gpu(li)
    assert status == 0
    y_ref, r = _oracle_y(li, from_planes=True)
    assert np.array_equal(call.route.ids.cpu().numpy(), r["ids"])
    _assert_close(y_ref, y)


@pytest.mark.parametrize("bits,T", [(4, 1), (3, 1), (8, 1), (5, 8), (6, 64), (8, 100)])
def test_ffn_back_to_back_calls(bits, T):
    """Thirty back-to-back calls of one 8x7B-shaped layer on the decode path:
    every call completes (no wait runs out) and returns the same bits (the
    combine order is fixed), and every token matches the oracle."""
    wl = synth.MIXTRAL_8X7B_SWEEP.with_(fixed_bits=bits, tokens=T)
    li = synth.layer_inputs(wl, device=DEV)
    sh = wl.shape
    stack = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, wl.parent_bits, wl.seed_bits, DEV)
    load_layer(stack, 0, li)
    stack.sync()
    call = MoECall(stack, T)
    opts = pw.pw_ffn_options()
    opts.path = pw.PW_PATH_DECODE
    first = None
    for _ in range(30):
        y = call(0, li.x, li.logits, options=opts)
        torch.cuda.synchronize()
        assert int(call.status.item()) == 0
        if first is None:
            first = y.clone()
        else:
            assert torch.equal(y, first)
    _check_rows(li, first.float().cpu().numpy(), list(range(T)))


def test_ffn_is_deterministic():
    li = synth.layer_inputs(synth.TINY_LAYER.with_(tokens=40))
    y1, s1, call, stack = _run_gpu(li)
    y2 = call(0, li.x.to(DEV), li.logits.to(DEV)).float().cpu().numpy()
    torch.cuda.synchronize()
    assert s1 == 0 and np.array_equal(y1, y2)


@pytest.mark.parametrize("path", [pw.PW_PATH_DECODE, pw.PW_PATH_PREFILL])
@pytest.mark.parametrize("H,I,E,k,T,bits", [
    (256, 256, 1, 1, 5, (3, 5)),          # single expert, k = 1
    (256, 512, 2, 2, 80, (8, 2)),         # 80 tokens per expert: several token tiles on the decode path
    (512, 768, 4, 2, 1, (4, 7)),          # one token
    (256, 2304, 3, 1, 9, (6, 3)),         # I below the 3072-column down split
    (256, 3200, 2, 1, 6, (5, 8)),         # I = 3072 + 128: a one-tile last down split
    (128, 6272, 2, 2, 3, (3, 4)),         # I = 2 * 3072 + 128, H of one strip
    (384, 640, 2, 2, 300, (5, 4)),        # odd strip counts, 300 tokens per expert (128-token tiles)
    (256, 512, 2, 1, 192, (8, 3)),        # 96 tokens per expert: the smallest batch on 128-token tiles
    (128, 384, 3, 3, 250, (7, 6)),        # every token to every expert: 250 per expert, a ragged last tile
])
def test_ffn_edge_shapes(H, I, E, k, T, bits, path):
    wl = synth.Workload("edge", synth.MoEShape(H, I, E, k), tokens=T, parent_bits=8, seed_bits=2, seed=H + I + T,
                        bits_mode="uniform_choice", bits_choices=bits)
    li = synth.layer_inputs(wl)
    opts = pw.pw_ffn_options()
    opts.path = path
    y, status, _, _ = _run_gpu(li, options=opts)
    assert status == 0
    y_ref, _ = _oracle_y(li)
    _assert_close(y_ref, y)


@pytest.mark.parametrize("path", [pw.PW_PATH_DECODE, pw.PW_PATH_PREFILL])
def test_ffn_tiny_workload_both_paths(path):
    li = synth.layer_inputs(synth.TINY_LAYER)
    opts = pw.pw_ffn_options()
    opts.path = path
    y, status, _, _ = _run_gpu(li, options=opts)
    assert status == 0
    y_ref, _ = _oracle_y(li, from_planes=True)
    _assert_close(y_ref, y)


def test_ffn_idle_expert_is_not_read():
    """An expert no token routes to contributes nothing and its blocks are not
    needed: leave them uncommitted and the call still succeeds."""
    wl = synth.TINY_LAYER.with_(tokens=12)
    li = synth.layer_inputs(wl)
    li.logits[:, 3] = -30.0          # expert 3 never chosen
    sh = wl.shape
    stack = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, wl.parent_bits, wl.seed_bits, DEV)
    load_layer(stack, 0, li, experts=[0, 1, 2])
    stack.sync()
    call = MoECall(stack, wl.tokens)
    y = call(0, li.x.to(DEV), li.logits.to(DEV)).float().cpu().numpy()
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0
    y_ref, _ = _oracle_y(li)
    _assert_close(y_ref, y)


def test_ffn_reports_uncommitted_routed_block():
    wl = synth.TINY_LAYER
    li = synth.layer_inputs(wl)
    sh = wl.shape
    stack = APLMoEStack(sh.hidden, sh.intermediate, sh.experts, sh.top_k, 1, wl.parent_bits, wl.seed_bits, DEV)
    load_layer(stack, 0, li, experts=[0, 1, 2])     # expert 3 is routed to but never committed
    stack.sync()
    call = MoECall(stack, wl.tokens)
    call(0, li.x.to(DEV), li.logits.to(DEV))
    torch.cuda.synchronize()
    assert int(call.status.item()) == pw.PW_ERR_NOT_RESIDENT


def test_ffn_bounded_wait_reports_timeout():
    """Test hook: one gate_up unit never signals completion, so the down
    units that need it wait out their (short) bound; the kernel returns with
    PW_ERR_TIMEOUT in the status word and the context stays usable."""
    li = synth.layer_inputs(synth.TINY_LAYER)
    opts = pw.pw_ffn_options()
    opts.flags = pw.PW_FFN_FLAG_TEST_DROP_ONE_ARRIVAL
    opts.wait_timeout_us = 20000
    _, status, call, _ = _run_gpu(li, options=opts)
    assert status == pw.PW_ERR_TIMEOUT
    call.status.zero_()
    y = call(0, li.x.to(DEV), li.logits.to(DEV)).float().cpu().numpy()
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0
    y_ref, _ = _oracle_y(li)
    _assert_close(y_ref, y)


# ---------------------------------------------------------------------------
# full-size workloads: every token, or a token set covering every (expert,
# slot) pair; the oracle runs one expert per host core
# ---------------------------------------------------------------------------
def _oracle_rows(li, tokens):
    """Oracle rows y[tokens] of the layer at its committed bitwidths, and the
    oracle's routing."""
    sh, P = li.wl.shape, li.wl.parent_bits
    lg = li.logits.cpu().numpy()
    r = apl.route_topk_shared(lg, sh.top_k, sh.shared) if sh.shared else apl.route_topk(lg, sh.top_k)
    experts = sorted({int(e) for e in r["ids"][tokens].ravel()})
    with oracle_parallel.ExpertFiles() as f:
        for e in experts:
            for u in (0, 1):
                q = li.bits[2 * e + u]
                f.add(e, u, li.idx[(e, u)].cpu().numpy(), li.luts[(e, u)][q].cpu().numpy(), q)
        y = oracle_parallel.layer_rows(f, li.x.cpu().numpy(), r["ids"], r["w"], sh.intermediate, P, tokens)
    return y, r


def _check_rows(li, y, tokens):
    """The GPU output rows `tokens` against the oracle; every (expert, slot)
    pair the batch routes to must be among them."""
    y_ref, r = _oracle_rows(li, tokens)
    ids = r["ids"]
    pairs_all = {(int(ids[t, j]), j) for t in range(ids.shape[0]) for j in range(ids.shape[1])}
    pairs = {(int(ids[t, j]), j) for t in tokens for j in range(ids.shape[1])}
    assert pairs == pairs_all
    assert np.all(np.isfinite(y[tokens]))
    _assert_close(y_ref, y[tokens])
    return r


def test_ffn_mixtral_8x7b_decode_mixed_bits():
    """The 8x7B decode layer with per-block bitwidths on 3..8: every one of
    the 32 tokens against the oracle."""
    wl = synth.MIXTRAL_8X7B_DECODE
    li = synth.layer_inputs(wl, device=DEV)
    y, status, call, _ = _run_gpu(li)
    assert status == 0
    r = _check_rows(li, y, list(range(wl.tokens)))
    assert np.array_equal(call.route.ids.cpu().numpy(), r["ids"])
    assert np.array_equal(call.route.perm.cpu().numpy(), r["perm"])


@pytest.mark.parametrize("b,T", [(3, 1), (8, 256), (5, 64), (4, 64), (6, 64), (3, 8)])
def test_ffn_mixtral_8x7b_uniform_sweep_points(b, T):
    """Uniform-bitwidth sweep points of the 8x7B layer, every token."""
    wl = synth.MIXTRAL_8X7B_SWEEP.with_(fixed_bits=b, tokens=T)
    li = synth.layer_inputs(wl, device=DEV, lut_bits=range(wl.seed_bits, b + 1))
    y, status, _, _ = _run_gpu(li)
    assert status == 0
    _check_rows(li, y, list(range(T)))


def test_ffn_mixtral_8x22b_prefill():
    """The 8x22B-shaped prefill layer: 4096 tokens, Zipf-skewed routing, hot
    experts at 8 bits and the rest at 3-4 bits (64-token tiles): tokens
    covering every (expert, slot) pair plus 40 random ones."""
    wl = synth.MIXTRAL_8X22B_PREFILL
    li = synth.layer_inputs(wl, device=DEV)
    y, status, call, _ = _run_gpu(li)
    assert status == 0
    r_ids = call.route.ids.cpu().numpy()
    toks = oracle_parallel.covering_tokens(r_ids, extra=40, seed=7)
    r = _check_rows(li, y, toks)
    assert np.array_equal(r_ids, r["ids"])
    assert np.array_equal(call.route.perm.cpu().numpy(), r["perm"])


# ---------------------------------------------------------------------------
# the CUDA-core instance (PW_KERNEL_CUDA_CORES): a split-K GEMV per unit
# ---------------------------------------------------------------------------
def _opts_cuda_cores(path=None):
    o = pw.pw_ffn_options()
    o.kernel = pw.PW_KERNEL_CUDA_CORES
    if path is not None:
        o.path = path
    return o


@pytest.mark.parametrize("path", [pw.PW_PATH_DECODE, pw.PW_PATH_PREFILL])
def test_cuda_core_kernel_tiny(path):
    li = synth.layer_inputs(synth.TINY_LAYER)
    y, status, call, _ = _run_gpu(li, options=_opts_cuda_cores(path))
    assert status == 0
    y_ref, r = _oracle_y(li, from_planes=True)
    assert np.array_equal(call.route.ids.cpu().numpy(), r["ids"])
    _assert_close(y_ref, y)


@pytest.mark.parametrize("b,T", [(3, 1), (8, 1), (5, 4), (3, 8)])
def test_cuda_core_kernel_mixtral_sweep_points(b, T):
    """Small decode batches of the 8x7B layer (one or two tokens per expert)
    on the CUDA cores, every token against the oracle."""
    wl = synth.MIXTRAL_8X7B_SWEEP.with_(fixed_bits=b, tokens=T)
    li = synth.layer_inputs(wl, device=DEV, lut_bits=range(wl.seed_bits, b + 1))
    y, status, _, _ = _run_gpu(li, options=_opts_cuda_cores())
    assert status == 0
    _check_rows(li, y, list(range(T)))


def test_cuda_core_kernel_mixed_bits_skewed_groups():
    """The decode layer with mixed bitwidths (up to ~14 tokens per expert, so
    many 2-token units per expert) on the CUDA cores; repeated calls return
    the same bits."""
    wl = synth.MIXTRAL_8X7B_DECODE
    li = synth.layer_inputs(wl, device=DEV)
    y, status, call, _ = _run_gpu(li, options=_opts_cuda_cores())
    assert status == 0
    y2 = call(0, li.x, li.logits, options=_opts_cuda_cores()).float().cpu().numpy()
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0 and np.array_equal(y, y2)
    _check_rows(li, y, list(range(wl.tokens)))


@pytest.mark.parametrize("H,I,E,k,T,bits", [(256, 2304, 3, 1, 9, (6, 3)), (128, 6272, 2, 2, 3, (3, 4)),
                                           (384, 640, 2, 2, 7, (5, 4))])
def test_cuda_core_kernel_edge_shapes(H, I, E, k, T, bits):
    wl = synth.Workload("edge", synth.MoEShape(H, I, E, k), tokens=T, parent_bits=8, seed_bits=2, seed=H + I + T,
                        bits_mode="uniform_choice", bits_choices=bits)
    li = synth.layer_inputs(wl)
    y, status, _, _ = _run_gpu(li, options=_opts_cuda_cores())
    assert status == 0
    y_ref, _ = _oracle_y(li)
    _assert_close(y_ref, y)
