"""Thin Python binding of libpw's C ABI (include/pw.h): same names, argument
marshalling only.  Every step of the path runs in libpw's CUDA kernels; there
is no Python or CPU fallback.  Tensors are torch tensors (device memory);
``stream`` defaults to torch's current CUDA stream.

Importing this module loads ``libpw.so`` from the package directory and fails
loudly if it is missing (build it with ``python -m any_precision_bit_pw_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpw.so")

PW_OK = 0
PW_ERR_INVALID_ARG = -1
PW_ERR_UNSUPPORTED = -2
PW_ERR_NOT_RESIDENT = -3
PW_ERR_CUDA = -4
PW_ERR_TIMEOUT = -5
PW_ERR_WORKSPACE = -6
PW_ERR_BUSY = -7
PW_PAGE_GPU, PW_PAGE_CPU, PW_PAGE_TO_CPU, PW_PAGE_TO_GPU = 1, 2, 4, 8


def PW_PAGE_LUT(b: int) -> int:
    return 8 + b

PW_LAYOUT_TILED = 1
PW_MAX_BITS = 8
PW_PATH_AUTO, PW_PATH_DECODE, PW_PATH_PREFILL = 0, 1, 2
PW_KERNEL_AUTO, PW_KERNEL_TENSOR, PW_KERNEL_CUDA_CORES = 0, 1, 2
PW_FFN_FLAG_TEST_DROP_ONE_ARRIVAL = 1
PW_FFN_FLAG_STRIP_COMBINE = 2

ERR_NAMES = {0: "PW_OK", -1: "PW_ERR_INVALID_ARG", -2: "PW_ERR_UNSUPPORTED", -3: "PW_ERR_NOT_RESIDENT",
             -4: "PW_ERR_CUDA", -5: "PW_ERR_TIMEOUT", -6: "PW_ERR_WORKSPACE", -7: "PW_ERR_BUSY"}

EXPORTS = (
    "pw_last_error", "pw_plane_bytes", "pw_pack_bitplanes", "pw_pack_lut", "pw_desc_bytes", "pw_page_table_create",
    "pw_page_table_destroy", "pw_page_table_attach_plane", "pw_page_table_attach_lut",
    "pw_page_table_set_desired", "pw_page_table_set_bits", "pw_page_table_get", "pw_page_table_bytes",
    "pw_page_table_resident_bytes", "pw_page_table_sync", "pw_moe_route_topk", "pw_moe_route_topk_shared",
    "pw_page_bytes", "pw_page_offload", "pw_page_reload", "pw_page_table_poll", "pw_page_table_take_released",
    "pw_page_state",
    "pw_moe_apl_ffn_workspace", "pw_moe_apl_ffn", "pw_moe_apl_ffn_ex", "pw_moe_apl_ffn_noalloc",
    "pw_moe_route_apl_ffn", "pw_moe_route_apl_ffn_ex", "pw_moe_route_apl_ffn_layers",
    "pw_unpack_indices",
    "pw_apl_linear",
)


class PwError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


class pw_block_info(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("parent_bits", ctypes.c_int32),
                ("seed_bits", ctypes.c_int32), ("layout", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class pw_ffn_options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("flags", ctypes.c_uint32), ("wait_timeout_us", ctypes.c_uint32),
                ("shared_experts", ctypes.c_int32), ("kernel", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]


_lib: Optional[ctypes.CDLL] = None
P, I32, I64, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libpw.so not built at {LIB_PATH}; run python -m any_precision_bit_pw_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "pw_last_error": (ctypes.c_char_p, []),
            "pw_plane_bytes": (SZ, [I64, I64, I32]),
            "pw_pack_bitplanes": (I32, [P, I64, I64, I32, ctypes.POINTER(P), I32, P]),
            "pw_pack_lut": (I32, [P, I64, I32, P, P]),
            "pw_desc_bytes": (SZ, [I32]),
            "pw_page_table_create": (I32, [ctypes.POINTER(P), I32, ctypes.POINTER(pw_block_info)]),
            "pw_page_table_destroy": (I32, [P]),
            "pw_page_table_attach_plane": (I32, [P, I32, I32, P]),
            "pw_page_table_attach_lut": (I32, [P, I32, I32, P]),
            "pw_page_table_set_desired": (I32, [P, I32, I32]),
            "pw_page_table_set_bits": (I32, [P, I32, I32, ctypes.POINTER(U64)]),
            "pw_page_table_get": (I32, [P, I32, ctypes.POINTER(I32), ctypes.POINTER(I32), ctypes.POINTER(U64)]),
            "pw_page_table_bytes": (I64, [P, I32, I32]),
            "pw_page_table_resident_bytes": (I64, [P]),
            "pw_page_table_sync": (I32, [P, P, SZ, P]),
            "pw_page_bytes": (I64, [P, I32, I32]),
            "pw_page_offload": (I32, [P, I32, I32, P, P]),
            "pw_page_reload": (I32, [P, I32, I32, P, P, P]),
            "pw_page_table_poll": (I32, [P, ctypes.POINTER(I32)]),
            "pw_page_table_take_released": (I32, [P, I32, ctypes.POINTER(U64)]),
            "pw_page_state": (I32, [P, I32, I32, ctypes.POINTER(I32), ctypes.POINTER(P), ctypes.POINTER(P)]),
            "pw_moe_route_topk": (I32, [P, I32, I32, I32, P, P, P, P, P, P, P]),
            "pw_moe_route_topk_shared": (I32, [P, I32, I32, I32, I32, P, P, P, P, P, P, P]),
            "pw_moe_apl_ffn_workspace": (SZ, [I32, I32, I32, I32, I32]),
            "pw_moe_apl_ffn": (I32, [P, I32, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, SZ, P, P, P]),
            "pw_moe_apl_ffn_ex": (I32, [P, I32, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, SZ, P, P,
                                        ctypes.POINTER(pw_ffn_options), P]),
            "pw_moe_apl_ffn_noalloc": (I32, [P, I32, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P]),
            "pw_moe_route_apl_ffn": (I32, [P, I32, P, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, SZ, P, P,
                                           P]),
            "pw_moe_route_apl_ffn_ex": (I32, [P, I32, P, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, SZ, P,
                                              P, ctypes.POINTER(pw_ffn_options), P]),
            "pw_moe_route_apl_ffn_layers": (I32, [P, I32, I32, P, P, I32, I32, I32, I32, I32, P, P, P, P, P, P, P,
                                                  SZ, P, P, ctypes.POINTER(pw_ffn_options), P]),
            "pw_unpack_indices": (I32, [P, I32, I32, P, P]),
            "pw_apl_linear": (I32, [P, I32, P, I32, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(rc: int) -> int:
    if rc != PW_OK:
        raise PwError(rc, pw_last_error())
    return rc


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: need a contiguous CUDA tensor of {dtype}, got {t.dtype} on {t.device}")


# ---------------------------------------------------------------------------
def pw_last_error() -> str:
    return lib().pw_last_error().decode(errors="replace")


def pw_plane_bytes(rows: int, cols: int, layout: int = PW_LAYOUT_TILED) -> int:
    return int(lib().pw_plane_bytes(rows, cols, layout))


def pw_pack_bitplanes(idx: torch.Tensor, parent_bits: int, planes: Sequence[torch.Tensor],
                      layout: int = PW_LAYOUT_TILED, stream=None) -> None:
    _dev(idx, torch.uint8, "idx")
    if len(planes) != parent_bits:
        raise ValueError("need one plane buffer per parent bit")
    arr = (P * parent_bits)(*[p.data_ptr() for p in planes])
    _check(lib().pw_pack_bitplanes(_ptr(idx), idx.shape[0], idx.shape[1], parent_bits, arr, layout,
                                   _stream(stream)))


def pw_pack_lut(lut: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """fp16 [rows][2^b] row-major LUT -> `out` (same size) in the tiled LUT layout."""
    _dev(lut, torch.float16, "lut")
    rows, C = lut.shape
    bits = C.bit_length() - 1
    if C != 1 << bits or not out.is_cuda or out.numel() * out.element_size() < rows * C * 2:
        raise ValueError("pack_lut: need lut [rows][2^b] and an output of the same size")
    _check(lib().pw_pack_lut(_ptr(lut), rows, bits, _ptr(out), _stream(stream)))


def pw_desc_bytes(n_blocks: int) -> int:
    return int(lib().pw_desc_bytes(n_blocks))


def pw_page_table_create(infos: Sequence[pw_block_info]) -> ctypes.c_void_p:
    arr = (pw_block_info * len(infos))(*infos)
    h = ctypes.c_void_p()
    _check(lib().pw_page_table_create(ctypes.byref(h), len(infos), arr))
    return h


def pw_page_table_destroy(t) -> None:
    _check(lib().pw_page_table_destroy(t))


def pw_page_table_attach_plane(t, block: int, plane: int, d_plane_ptr: int) -> None:
    _check(lib().pw_page_table_attach_plane(t, block, plane, ctypes.c_void_p(d_plane_ptr)))


def pw_page_table_attach_lut(t, block: int, bits: int, d_lut_ptr: int) -> None:
    _check(lib().pw_page_table_attach_lut(t, block, bits, ctypes.c_void_p(d_lut_ptr)))


def pw_page_table_set_desired(t, block: int, d: int) -> None:
    _check(lib().pw_page_table_set_desired(t, block, d))


def pw_page_table_set_bits(t, block: int, q: int) -> int:
    """Returns the released-page mask (bit p: plane p; bit 8+b: LUT b)."""
    m = U64(0)
    _check(lib().pw_page_table_set_bits(t, block, q, ctypes.byref(m)))
    return int(m.value)


def pw_page_table_get(t, block: int):
    q, d, m = I32(0), I32(0), U64(0)
    _check(lib().pw_page_table_get(t, block, ctypes.byref(q), ctypes.byref(d), ctypes.byref(m)))
    return int(q.value), int(d.value), int(m.value)


def pw_page_table_bytes(t, block: int, b: int) -> int:
    return int(lib().pw_page_table_bytes(t, block, b))


def pw_page_table_resident_bytes(t) -> int:
    return int(lib().pw_page_table_resident_bytes(t))


def pw_page_table_sync(t, d_desc: torch.Tensor, stream=None) -> None:
    _check(lib().pw_page_table_sync(t, _ptr(d_desc), d_desc.numel() * d_desc.element_size(), _stream(stream)))


def pw_page_bytes(t, block: int, page: int) -> int:
    return int(lib().pw_page_bytes(t, block, page))


def pw_page_offload(t, block: int, page: int, host: torch.Tensor, stream=None) -> None:
    """Start copying a GPU-resident page into `host` (pinned, >= pw_page_bytes bytes)."""
    if host.is_cuda or host.numel() * host.element_size() < pw_page_bytes(t, block, page):
        raise ValueError("offload: need a host tensor of at least the page's bytes")
    _check(lib().pw_page_offload(t, block, page, _ptr(host), _stream(stream)))


def pw_page_reload(t, block: int, page: int, host: Optional[torch.Tensor], dev: torch.Tensor, stream=None) -> None:
    """Start copying a page from `host` (None: the page's own host copy) into `dev`."""
    if not dev.is_cuda or dev.numel() * dev.element_size() < pw_page_bytes(t, block, page):
        raise ValueError("reload: need a device tensor of at least the page's bytes")
    _check(lib().pw_page_reload(t, block, page, _ptr(host), _ptr(dev), _stream(stream)))


def pw_page_table_poll(t) -> int:
    """Advance finished transfers; returns the number still in flight."""
    n = I32(0)
    _check(lib().pw_page_table_poll(t, ctypes.byref(n)))
    return int(n.value)


def pw_page_table_take_released(t, block: int) -> int:
    m = U64(0)
    _check(lib().pw_page_table_take_released(t, block, ctypes.byref(m)))
    return int(m.value)


def pw_page_state(t, block: int, page: int):
    """(state bits, attached device address or 0, host address or 0)."""
    st, d, h = I32(0), P(), P()
    _check(lib().pw_page_state(t, block, page, ctypes.byref(st), ctypes.byref(d), ctypes.byref(h)))
    return int(st.value), int(d.value or 0), int(h.value or 0)


def pw_moe_route_topk(logits: torch.Tensor, k: int, ids: torch.Tensor, w: torch.Tensor, offsets: torch.Tensor,
                      perm: torch.Tensor, inv_perm: torch.Tensor, mass_accum: Optional[torch.Tensor] = None,
                      stream=None) -> None:
    _dev(logits, torch.float32, "logits")
    T, E = logits.shape
    _check(lib().pw_moe_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _ptr(offsets), _ptr(perm),
                                   _ptr(inv_perm), _ptr(mass_accum), _stream(stream)))


def pw_moe_route_topk_shared(logits: torch.Tensor, k: int, shared: int, ids: torch.Tensor, w: torch.Tensor,
                             offsets: torch.Tensor, perm: torch.Tensor, inv_perm: torch.Tensor,
                             mass_accum: Optional[torch.Tensor] = None, stream=None) -> None:
    """Top-k routing plus `shared` always-on experts (ids E..E+S-1, weight 1)."""
    _dev(logits, torch.float32, "logits")
    T, E = logits.shape
    _check(lib().pw_moe_route_topk_shared(_ptr(logits), T, E, k, shared, _ptr(ids), _ptr(w), _ptr(offsets),
                                          _ptr(perm), _ptr(inv_perm), _ptr(mass_accum), _stream(stream)))


def pw_moe_apl_ffn_workspace(T: int, H: int, I: int, E: int, k: int) -> int:
    return int(lib().pw_moe_apl_ffn_workspace(T, H, I, E, k))


def pw_moe_apl_ffn(d_desc: torch.Tensor, layer: int, x: torch.Tensor, I: int, E: int, k: int,
                   ids: Optional[torch.Tensor], w: torch.Tensor, offsets: torch.Tensor, perm: torch.Tensor,
                   inv_perm: torch.Tensor, ws: torch.Tensor, y: torch.Tensor, status: torch.Tensor,
                   options: Optional[pw_ffn_options] = None, stream=None) -> None:
    _dev(x, torch.float16, "x")
    _dev(y, torch.float16, "y")
    T, H = x.shape
    args = (_ptr(d_desc), layer, _ptr(x), T, H, I, E, k, _ptr(ids), _ptr(w), _ptr(offsets), _ptr(perm),
            _ptr(inv_perm), _ptr(ws), ws.numel() * ws.element_size(), _ptr(y), _ptr(status))
    if options is None:
        _check(lib().pw_moe_apl_ffn(*args, _stream(stream)))
    else:
        _check(lib().pw_moe_apl_ffn_ex(*args, ctypes.byref(options), _stream(stream)))


def pw_moe_route_apl_ffn(d_desc: torch.Tensor, layer: int, x: torch.Tensor, logits: torch.Tensor, I: int, E: int,
                         k: int, ids: torch.Tensor, w: torch.Tensor, offsets: torch.Tensor, perm: torch.Tensor,
                         inv_perm: torch.Tensor, mass_accum: Optional[torch.Tensor], ws: torch.Tensor,
                         y: torch.Tensor, status: torch.Tensor, options: Optional[pw_ffn_options] = None,
                         stream=None) -> None:
    """Routing and the fused expert layer (the routing arrays are outputs):
    one launch for batches one warp routes (at most 32 tokens, 8 experts and
    4 slots per token), else a routing launch and the fused launch."""
    _dev(x, torch.float16, "x")
    _dev(y, torch.float16, "y")
    _dev(logits, torch.float32, "logits")
    T, H = x.shape
    if tuple(logits.shape) != (T, E):
        raise ValueError(f"logits: need shape ({T}, {E}), got {tuple(logits.shape)}")
    args = (_ptr(d_desc), layer, _ptr(x), _ptr(logits), T, H, I, E, k, _ptr(ids), _ptr(w), _ptr(offsets),
            _ptr(perm), _ptr(inv_perm), _ptr(mass_accum), _ptr(ws), ws.numel() * ws.element_size(), _ptr(y),
            _ptr(status))
    if options is None:
        _check(lib().pw_moe_route_apl_ffn(*args, _stream(stream)))
    else:
        _check(lib().pw_moe_route_apl_ffn_ex(*args, ctypes.byref(options), _stream(stream)))


def pw_moe_route_apl_ffn_layers(d_desc: torch.Tensor, layer0: int, x: torch.Tensor, logits: torch.Tensor, I: int,
                                E: int, k: int, ids: torch.Tensor, w: torch.Tensor, offsets: torch.Tensor,
                                perm: torch.Tensor, inv_perm: torch.Tensor, mass_accum: Optional[torch.Tensor],
                                ws: torch.Tensor, y: torch.Tensor, status: torch.Tensor,
                                options: Optional[pw_ffn_options] = None, stream=None) -> None:
    """Routing and the fused expert layer of L independent layers in one
    launch: x [L][T][H], logits [L][T][E], y [L][T][H]; the routing arrays
    are outputs in the layers' concatenated index space (see pw.h)."""
    _dev(x, torch.float16, "x")
    _dev(y, torch.float16, "y")
    _dev(logits, torch.float32, "logits")
    L, T, H = x.shape
    if tuple(logits.shape) != (L, T, E) or tuple(y.shape[:2]) != (L, T) or y.shape[2] != H:
        raise ValueError(f"layers call: x {tuple(x.shape)}, logits {tuple(logits.shape)}, y {tuple(y.shape)}")
    opts = options if options is not None else pw_ffn_options()
    _check(lib().pw_moe_route_apl_ffn_layers(_ptr(d_desc), layer0, L, _ptr(x), _ptr(logits), T, H, I, E, k, _ptr(ids),
                                             _ptr(w), _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(mass_accum),
                                             _ptr(ws), ws.numel() * ws.element_size(), _ptr(y), _ptr(status),
                                             ctypes.byref(opts), _stream(stream)))


PW_NOALLOC_SCRATCH_BYTES = 32 << 20


def pw_moe_apl_ffn_noalloc(d_desc: torch.Tensor, layer: int, x: torch.Tensor, I: int, E: int, k: int,
                           ids: Optional[torch.Tensor], w: torch.Tensor, offsets: torch.Tensor,
                           perm: torch.Tensor, inv_perm: torch.Tensor, y: torch.Tensor, status: torch.Tensor,
                           stream=None) -> None:
    """pw_moe_apl_ffn without a caller workspace: libpw's built-in scratch
    array is used instead (see include/pw.h for its size and sharing rules)."""
    _dev(x, torch.float16, "x")
    _dev(y, torch.float16, "y")
    T, H = x.shape
    _check(lib().pw_moe_apl_ffn_noalloc(_ptr(d_desc), layer, _ptr(x), T, H, I, E, k, _ptr(ids), _ptr(w),
                                        _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(y), _ptr(status),
                                        _stream(stream)))


def pw_unpack_indices(t, block: int, b: int, out: torch.Tensor, stream=None) -> None:
    _dev(out, torch.uint8, "out")
    _check(lib().pw_unpack_indices(t, block, b, _ptr(out), _stream(stream)))


def pw_apl_linear(t, block: int, x: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _dev(x, torch.float16, "x")
    _dev(out, torch.float32, "out")
    _check(lib().pw_apl_linear(t, block, _ptr(x), x.shape[0], _ptr(out), _stream(stream)))
