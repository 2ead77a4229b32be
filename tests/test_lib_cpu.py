"""Host-side checks of libpw that need no GPU: the library loads, exports
every call the header declares, and the page table (pure host state) follows
the ordering and accounting rules of the PagedWeight arXiv text (§3.1, Eq. 3)."""
import os
import re

import pytest

from oracle import apl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pw = pytest.importorskip("any_precision_bit_pw_gb300.pw")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(pw.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return pw.lib()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "pw.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pw_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = _header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n
    assert set(pw.EXPORTS) == set(names)


def test_plane_bytes(L):
    assert pw.pw_plane_bytes(28672, 4096) == 14_680_064
    assert pw.pw_plane_bytes(4096, 14336) == 7_340_032
    assert pw.pw_plane_bytes(1024, 256) == 32_768
    assert pw.pw_plane_bytes(8, 256) == 0
    assert pw.pw_plane_bytes(16, 128) == 0
    assert pw.pw_plane_bytes(16, 256, layout=0) == 0


def _table(blocks=2, rows=128, cols=512, P=8, S=3):
    infos = [pw.pw_block_info(rows, cols, P, S, pw.PW_LAYOUT_TILED, 0) for _ in range(blocks)]
    return pw.pw_page_table_create(infos)


FAKE = 0x7F0000000000  # never dereferenced: the table only stores pointers


def test_page_table_raise_needs_resident_pages(L):
    t = _table()
    try:
        with pytest.raises(pw.PwError) as e:
            pw.pw_page_table_set_bits(t, 0, 4)
        assert e.value.code == pw.PW_ERR_NOT_RESIDENT
        for p in range(4):
            pw.pw_page_table_attach_plane(t, 0, p, FAKE + 0x1000 * p)
        with pytest.raises(pw.PwError) as e:           # LUTs 3 and 4 still missing
            pw.pw_page_table_set_bits(t, 0, 4)
        assert e.value.code == pw.PW_ERR_NOT_RESIDENT
        pw.pw_page_table_attach_lut(t, 0, 3, FAKE + 0x100000)
        pw.pw_page_table_attach_lut(t, 0, 4, FAKE + 0x200000)
        assert pw.pw_page_table_set_bits(t, 0, 4) == 0
        assert pw.pw_page_table_get(t, 0)[0] == 4
        assert pw.pw_page_table_get(t, 1)[0] == 0
    finally:
        pw.pw_page_table_destroy(t)


def test_page_table_lowering_releases_only_pages_above(L):
    t = _table()
    try:
        for p in range(8):
            pw.pw_page_table_attach_plane(t, 0, p, FAKE + 0x1000 * p)
        for b in range(3, 9):
            pw.pw_page_table_attach_lut(t, 0, b, FAKE + 0x100000 * b)
        assert pw.pw_page_table_set_bits(t, 0, 8) == 0
        mask = pw.pw_page_table_set_bits(t, 0, 5)
        assert mask == (0b11100000 | (1 << (8 + 6)) | (1 << (8 + 7)) | (1 << (8 + 8)))
        q, d, res = pw.pw_page_table_get(t, 0)
        assert q == 5
        assert res == (0b00011111 | sum(1 << (8 + b) for b in (3, 4, 5)))
        # raising again needs the released pages back (reload, then raise)
        with pytest.raises(pw.PwError):
            pw.pw_page_table_set_bits(t, 0, 6)
        pw.pw_page_table_attach_plane(t, 0, 5, FAKE + 0x5000)
        pw.pw_page_table_attach_lut(t, 0, 6, FAKE + 0x600000)
        assert pw.pw_page_table_set_bits(t, 0, 6) == 0
        # below the seed bitwidth is not a supported bitwidth
        with pytest.raises(pw.PwError) as e:
            pw.pw_page_table_set_bits(t, 0, 2)
        assert e.value.code == pw.PW_ERR_INVALID_ARG
    finally:
        pw.pw_page_table_destroy(t)


def test_page_table_bytes_match_eq3(L):
    rows, cols, S = 28672, 4096, 3
    t = _table(blocks=3, rows=rows, cols=cols, S=S)
    try:
        for b in range(S, 9):
            assert pw.pw_page_table_bytes(t, 1, b) == apl.page_bytes(rows, cols, S, b)
        assert pw.pw_page_table_bytes(t, 1, 2) == -1
        assert pw.pw_page_table_bytes(t, 7, 4) == -1
        assert pw.pw_page_table_resident_bytes(t) == 0
        for p in range(8):
            pw.pw_page_table_attach_plane(t, 2, p, FAKE + 0x1000 * p)
        for b in range(3, 9):
            pw.pw_page_table_attach_lut(t, 2, b, FAKE + 0x100000 * b)
        pw.pw_page_table_set_bits(t, 2, 8)
        before = pw.pw_page_table_resident_bytes(t)
        pw.pw_page_table_set_bits(t, 2, 4)
        after = pw.pw_page_table_resident_bytes(t)
        assert before - after == apl.released_bytes(rows, cols, S, 8, 4)
    finally:
        pw.pw_page_table_destroy(t)


def test_page_table_argument_errors(L):
    with pytest.raises(pw.PwError):
        pw.pw_page_table_create([pw.pw_block_info(8, 256, 8, 3, 1, 0)])        # rows % 16
    with pytest.raises(pw.PwError):
        pw.pw_page_table_create([pw.pw_block_info(16, 256, 8, 9, 1, 0)])       # seed > parent
    t = _table()
    try:
        with pytest.raises(pw.PwError):
            pw.pw_page_table_attach_plane(t, 0, 8, FAKE)                        # plane >= parent
        with pytest.raises(pw.PwError):
            pw.pw_page_table_attach_plane(t, 0, 0, FAKE + 4)                    # misaligned
        with pytest.raises(pw.PwError):
            pw.pw_page_table_attach_lut(t, 0, 2, FAKE)                          # below seed
        with pytest.raises(pw.PwError):
            pw.pw_page_table_set_desired(t, 0, 9)
        pw.pw_page_table_set_desired(t, 0, 5)
        assert pw.pw_page_table_get(t, 0)[1] == 5
        with pytest.raises(pw.PwError) as e:
            pw.pw_page_table_get(t, 2)
        assert "out of range" in str(e.value)
    finally:
        pw.pw_page_table_destroy(t)


def test_workspace_and_host_validation(L):
    assert pw.pw_moe_apl_ffn_workspace(32, 4096, 14336, 8, 2) > 32 * 2 * 14336 * 2
    assert pw.pw_moe_apl_ffn_workspace(32, 4000, 14336, 8, 2) == 0       # H not a multiple of 128
    assert pw.pw_moe_apl_ffn_workspace(32, 4096, 14336, 8, 9) == 0       # k > E
    # argument errors are caught on the host before any CUDA call
    rc = L.pw_moe_route_topk(None, 4, 0, 1, None, None, None, None, None, None, None)
    assert rc == pw.PW_ERR_UNSUPPORTED
    rc = L.pw_moe_route_topk(None, 4, 8, 9, None, None, None, None, None, None, None)
    assert rc == pw.PW_ERR_UNSUPPORTED
    assert "k <=" in pw.pw_last_error()


def test_routed_ffn_checks_arguments_before_any_launch(L):
    """The routed layer call rejects missing logits and routing outputs on the
    host (no device is touched)."""
    rc = L.pw_moe_route_apl_ffn(None, 0, None, None, 4, 128, 128, 4, 2, None, None, None, None, None, None,
                                None, 0, None, None, None)
    assert rc == pw.PW_ERR_INVALID_ARG and "logits" in pw.pw_last_error()
    fake = 0x7F0000000000
    rc = L.pw_moe_route_apl_ffn(fake, 0, fake, fake, 4, 128, 128, 4, 2, None, fake, None, fake, fake, None,
                                fake, 1 << 20, fake, fake, None)
    assert rc == pw.PW_ERR_INVALID_ARG and "ids and offsets" in pw.pw_last_error()


def test_page_movement_host_checks(L):
    """Page ids, sizes and the checks pw_page_offload / pw_page_reload make
    before any copy is enqueued (§3.1 page states)."""
    import ctypes
    t = _table(blocks=1, rows=128, cols=512, P=8, S=3)
    try:
        assert pw.pw_page_bytes(t, 0, 0) == 128 * 512 // 8
        assert pw.pw_page_bytes(t, 0, 7) == 128 * 512 // 8
        assert pw.pw_page_bytes(t, 0, pw.PW_PAGE_LUT(3)) == 128 * 8 * 2
        assert pw.pw_page_bytes(t, 0, pw.PW_PAGE_LUT(8)) == 128 * 256 * 2
        for bad in (-1, 8 + 2, 17):
            assert pw.pw_page_bytes(t, 0, bad) == -1
        assert pw.pw_page_state(t, 0, 2) == (0, 0, 0)
        # offload of a page that is not GPU-resident
        rc = L.pw_page_offload(t, 0, 2, ctypes.c_void_p(FAKE), None)
        assert rc == pw.PW_ERR_NOT_RESIDENT
        # reload without a host copy, and into a misaligned buffer
        rc = L.pw_page_reload(t, 0, 2, None, ctypes.c_void_p(FAKE), None)
        assert rc == pw.PW_ERR_NOT_RESIDENT
        rc = L.pw_page_reload(t, 0, 2, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + 4), None)
        assert rc == pw.PW_ERR_INVALID_ARG
        # an attached page is GPU-resident; reloading into it is refused
        pw.pw_page_table_attach_plane(t, 0, 2, FAKE)
        assert pw.pw_page_state(t, 0, 2) == (pw.PW_PAGE_GPU, FAKE, 0)
        rc = L.pw_page_reload(t, 0, 2, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), None)
        assert rc == pw.PW_ERR_INVALID_ARG
        # nothing in flight: poll touches no device and reports 0
        assert pw.pw_page_table_poll(t) == 0
        assert pw.pw_page_table_take_released(t, 0) == 0
    finally:
        pw.pw_page_table_destroy(t)


def test_noalloc_accepts_exactly_the_sizes_whose_path_fits(L):
    """pw_moe_apl_ffn_noalloc takes a call when the workspace of the path the
    call runs on fits its fixed array.  For the Mixtral-8x7B shape at top-2
    the decode path (below 48 assignments per expert) fits up to 141 tokens,
    the prefill path from 192 up to 315 tokens; the size check comes before
    anything else that needs a GPU, so the rejections are seen here."""
    def rc(T):
        return L.pw_moe_apl_ffn_noalloc(None, 0, None, T, 4096, 14336, 8, 2, None, None, None, None, None,
                                        None, None, None)
    for T in (1, 32, 141, 192, 315):
        assert rc(T) != pw.PW_ERR_WORKSPACE, T
    for T in (142, 191, 316, 4096):
        assert rc(T) == pw.PW_ERR_WORKSPACE, T
        assert "scratch" in pw.pw_last_error()


def test_layers_call_checks_sizes_before_any_launch(L):
    def rc(nl, E=8, T=128):
        return L.pw_moe_route_apl_ffn_layers(None, 0, nl, None, None, T, 4096, 14336, E, 2, None, None, None, None,
                                             None, None, None, 0, None, None, None, None)
    assert rc(33) == pw.PW_ERR_UNSUPPORTED            # 33 layers x 8 experts > 256
    assert "exceed" in pw.pw_last_error()
    assert rc(0) == pw.PW_ERR_INVALID_ARG
    assert rc(32) == pw.PW_ERR_INVALID_ARG           # sizes fine: the NULL arguments are next
    assert rc(2, E=200) == pw.PW_ERR_UNSUPPORTED
