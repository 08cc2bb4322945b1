"""Thin ctypes binding over libqmoe.so (declared in include/qmoe.h).

Argument marshalling only: every function passes device pointers of torch
tensors, the sizes and the current CUDA stream to the C entry point of the
same name and raises QmoeError on a non-zero status.  There is no fallback:
when the CUDA library is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmoe.so")

SCHEME_ID = {"w4a16": 0, "mxfp4": 1, "w8a8": 2, "w4a8": 3}
DEV_BAD_EXPERT_ID = 1
DEV_WAIT_TIMEOUT = 2


class QmoeError(RuntimeError):
    pass


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("k", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32)]


class TileRule(ctypes.Structure):
    """qmoe_tile_rule: dims with these H, I, E, k (0 = any) and t_min <= T <= t_max use token tile nmax."""
    _fields_ = [("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("t_min", ctypes.c_int64), ("t_max", ctypes.c_int64), ("nmax", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_DP = ctypes.POINTER(Dims)

# name -> (argtypes, restype)
SIGNATURES = {
    "qmoe_status_str": ([_i32], ctypes.c_char_p),
    "qmoe_version": ([], ctypes.c_char_p),
    "qmoe_workspace_bytes": ([_DP], _sz),
    "qmoe_align_sort": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_align_sort_static_scratch": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "qmoe_quant_act_mxfp8": ([_i64, _i64, _vp, _vp, _vp, _vp], _i32),
    "qmoe_quant_rows_int8_bf16": ([_i64, _i64, _vp, _vp, _vp, _vp], _i32),
    "qmoe_quant_rows_int8_f32": ([_i64, _i64, _vp, _vp, _vp, _vp], _i32),
    "qmoe_mx_scales_packed_bytes": ([_i64, _i64], _sz),
    "qmoe_fp4_weights_packed_bytes": ([_i64, _i64], _sz),
    "qmoe_prepack_fp4_weights": ([_i64, _i64, _vp, _vp, _vp], _i32),
    "qmoe_prepack_mx_scales": ([_i64, _i64, _vp, _vp, _vp], _i32),
    "qmoe_int4_weights_packed_bytes": ([_i64, _i64], _sz),
    "qmoe_prepack_int4_weights": ([_i64, _i64, _vp, _vp, _vp, _vp], _i32),
    "qmoe_w4a16_x_tiles_bytes": ([_DP], _sz),
    "qmoe_w4a16_h_tiles_bytes": ([_DP], _sz),
    "qmoe_w4a16_h16_tiles_bytes": ([_DP], _sz),
    "qmoe_w4a16_h_to_f16": ([_DP, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_permute_x_f16": ([_DP, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_gemm1_swiglu_w4a16": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_mx_tiles_bytes": ([_DP, _i64], _sz),
    "qmoe_permute_quant_mxfp8": ([_DP, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_gemm1_swiglu_mxfp4": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_gemm1_swiglu_mxfp4_gather": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_mx_layer_gathers": ([_DP], _i32),
    "qmoe_forward_launches": ([_DP, _i32], _i32),
    "qmoe_w8a8_tiles_bytes": ([_DP, _i64], _sz),
    "qmoe_permute_quant_int8": ([_DP, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_quant_tiles_int8_f32": ([_DP, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_gemm1_swiglu_w8a8": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_gemm2_w4a16": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_gemm2_mxfp4": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_gemm2_w8a8": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_set_tile_rules": ([ctypes.POINTER(TileRule), _i32], _i32),
    "qmoe_tile_nmax": ([_DP], _i32),
    "qmoe_gemm1_swiglu_w4a8": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_gemm2_w4a8": ([_DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
    "qmoe_combine": ([_DP, _vp, _vp, _vp, _vp, _vp], _i32),
    "qmoe_forward_workspace_bytes": ([_DP, _i32], _sz),
    "qmoe_moe_forward": ([_i32, _DP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i32),
}

_lib = None


def lib():
    """Load libqmoe.so (raises when it is missing: there is no CPU path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise QmoeError(f"{LIB_PATH} is not built; run quantized_mixture_experts_moe_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        # the tuned token-tile table shipped beside the library (QMOE_TILE_TABLE: another
        # file, or "none" for the built-in rule alone)
        path = os.environ.get("QMOE_TILE_TABLE", TILE_TABLE_PATH)
        if path != "none" and os.path.exists(path):
            set_tile_rules(read_tile_table(path))
    return _lib


TILE_TABLE_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tile_table.csv")
TILE_TABLE_FIELDS = ("scheme", "H", "I", "E", "k", "t_min", "t_max", "nmax")


def read_tile_table(path):
    """Rules from a tile-table CSV (header row; one rule per line, first match wins).  The
    scheme column records what the row was measured on; the library's rule is per shape."""
    import csv

    with open(path) as f:
        rows = [r for r in csv.DictReader(line for line in f if not line.startswith("#"))]
    return [dict(H=int(r["H"]), I=int(r["I"]), E=int(r["E"]), k=int(r["k"]), t_min=int(r["t_min"]),
                 t_max=int(r["t_max"]), nmax=int(r["nmax"])) for r in rows]


def set_tile_rules(rules):
    """Replace the library's token-tile table (a list of dicts with H, I, E, k, t_min, t_max, nmax)."""
    arr = (TileRule * max(1, len(rules)))()
    for i, r in enumerate(rules):
        arr[i] = TileRule(r.get("H", 0), r.get("I", 0), r.get("E", 0), r.get("k", 0), r.get("t_min", 0),
                          r.get("t_max", 2**62), r["nmax"], 0)
    _check(lib().qmoe_set_tile_rules(arr, len(rules)), "qmoe_set_tile_rules")


def tile_nmax(d: Dims) -> int:
    """The token tile (16, 112 or 224) the library uses for dims d."""
    return int(lib().qmoe_tile_nmax(ctypes.byref(d)))


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise QmoeError("qmoe kernels take device tensors")
    if not t.is_contiguous():
        raise QmoeError("qmoe kernels take contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, name: str):
    if rc != 0:
        raise QmoeError(f"{name} failed: {rc} ({lib().qmoe_status_str(rc).decode()})")


def dims(T, k, H, I, E) -> Dims:
    return Dims(T, k, H, I, E)


def status_str(code: int) -> str:
    return lib().qmoe_status_str(code).decode()


def version() -> str:
    return lib().qmoe_version().decode()


def workspace_bytes(d: Dims) -> int:
    return int(lib().qmoe_workspace_bytes(ctypes.byref(d)))


def forward_workspace_bytes(d: Dims, scheme: str) -> int:
    return int(lib().qmoe_forward_workspace_bytes(ctypes.byref(d), SCHEME_ID[scheme]))


def qmoe_align_sort(d, topk_ids, counts, offsets, sorted_pair_ids, pair_slot, dev_status, ws, stream=None):
    rc = lib().qmoe_align_sort(ctypes.byref(d), _ptr(topk_ids), _ptr(counts), _ptr(offsets), _ptr(sorted_pair_ids),
                               _ptr(pair_slot), _ptr(dev_status), _ptr(ws), ws.numel() * ws.element_size(),
                               _stream(stream))
    _check(rc, "qmoe_align_sort")


STATIC_SCRATCH_BYTES = 1 << 20


def qmoe_align_sort_static_scratch(d, topk_ids, counts, offsets, sorted_pair_ids, pair_slot, dev_status,
                                   stream=None):
    """The routing sort with the library's built-in scratch (no workspace)."""
    rc = lib().qmoe_align_sort_static_scratch(ctypes.byref(d), _ptr(topk_ids), _ptr(counts), _ptr(offsets),
                                              _ptr(sorted_pair_ids), _ptr(pair_slot), _ptr(dev_status),
                                              _stream(stream))
    _check(rc, "qmoe_align_sort_static_scratch")


def qmoe_quant_act_mxfp8(x_bf16, x_q, x_s, stream=None):
    rows, cols = x_bf16.shape
    _check(lib().qmoe_quant_act_mxfp8(rows, cols, _ptr(x_bf16), _ptr(x_q), _ptr(x_s), _stream(stream)),
           "qmoe_quant_act_mxfp8")


def qmoe_quant_rows_int8_bf16(x, q, s, stream=None):
    rows, cols = x.shape
    _check(lib().qmoe_quant_rows_int8_bf16(rows, cols, _ptr(x), _ptr(q), _ptr(s), _stream(stream)),
           "qmoe_quant_rows_int8_bf16")


def qmoe_quant_rows_int8_f32(x, q, s, stream=None):
    rows, cols = x.shape
    _check(lib().qmoe_quant_rows_int8_f32(rows, cols, _ptr(x), _ptr(q), _ptr(s), _stream(stream)),
           "qmoe_quant_rows_int8_f32")


def _ws(ws):
    return _ptr(ws), (0 if ws is None else ws.numel() * ws.element_size())


def mx_scales_packed_bytes(rows: int, K: int) -> int:
    return int(lib().qmoe_mx_scales_packed_bytes(rows, K))


def qmoe_prepack_mx_scales(s_rowmajor, s_packed, rows: int, K: int, stream=None):
    _check(lib().qmoe_prepack_mx_scales(rows, K, _ptr(s_rowmajor), _ptr(s_packed), _stream(stream)),
           "qmoe_prepack_mx_scales")


def fp4_weights_packed_bytes(rows: int, K: int) -> int:
    return int(lib().qmoe_fp4_weights_packed_bytes(rows, K))


def qmoe_prepack_fp4_weights(w_rowmajor, w_packed, rows: int, K: int, stream=None):
    _check(lib().qmoe_prepack_fp4_weights(rows, K, _ptr(w_rowmajor), _ptr(w_packed), _stream(stream)),
           "qmoe_prepack_fp4_weights")


def prepack_fp4_weights(w_rowmajor, K: int, stream=None):
    """Packed 4-bit weights [..., K/2] (rows = all leading dims) -> tile-major byte tensor."""
    rows = w_rowmajor.numel() // (K // 2)
    out = torch.empty(max(fp4_weights_packed_bytes(rows, K), 16), dtype=torch.uint8, device=w_rowmajor.device)
    qmoe_prepack_fp4_weights(w_rowmajor.contiguous(), out, rows, K, stream)
    return out


def prepack_mxfp4(w1, w1_s, w2, w2_s, H: int, I: int, stream=None):
    """All four MXFP4 weight tensors in the form the GEMMs take."""
    return (prepack_fp4_weights(w1, H, stream), prepack_mx_scales(w1_s, H, stream),
            prepack_fp4_weights(w2, I, stream), prepack_mx_scales(w2_s, I, stream))


def prepack_mx_scales(s_rowmajor, K: int, stream=None):
    """E8M0 scales [..., K/32] (rows = all leading dims) -> packed byte tensor."""
    rows = s_rowmajor.numel() // (K // 32)
    out = torch.empty(max(mx_scales_packed_bytes(rows, K), 16), dtype=torch.uint8, device=s_rowmajor.device)
    qmoe_prepack_mx_scales(s_rowmajor.contiguous(), out, rows, K, stream)
    return out


def int4_weights_packed_bytes(rows: int, K: int) -> int:
    return int(lib().qmoe_int4_weights_packed_bytes(rows, K))


def qmoe_prepack_int4_weights(w_rowmajor, s_fp16, packed, rows: int, K: int, stream=None):
    _check(lib().qmoe_prepack_int4_weights(rows, K, _ptr(w_rowmajor), _ptr(s_fp16), _ptr(packed), _stream(stream)),
           "qmoe_prepack_int4_weights")


def prepack_int4_weights(w_rowmajor, s_fp16, K: int, stream=None):
    """int4 codes [..., K/2] + fp16 scales [..., K/32] (rows = all leading dims) -> packed byte tensor."""
    rows = w_rowmajor.numel() // (K // 2)
    out = torch.empty(max(int4_weights_packed_bytes(rows, K), 16), dtype=torch.uint8, device=w_rowmajor.device)
    qmoe_prepack_int4_weights(w_rowmajor.contiguous(), s_fp16.contiguous(), out, rows, K, stream)
    return out


def prepack_w4a16(w1, w1_s, w2, w2_s, H: int, I: int, stream=None):
    """Both W4A16 weight tensors (codes with their scales) in the form the GEMMs take."""
    return prepack_int4_weights(w1, w1_s, H, stream), prepack_int4_weights(w2, w2_s, I, stream)


def w4a16_x_tiles_bytes(d: Dims) -> int:
    return int(lib().qmoe_w4a16_x_tiles_bytes(ctypes.byref(d)))


def w4a16_h_tiles_bytes(d: Dims) -> int:
    return int(lib().qmoe_w4a16_h_tiles_bytes(ctypes.byref(d)))


def w4a16_h16_tiles_bytes(d: Dims) -> int:
    return int(lib().qmoe_w4a16_h16_tiles_bytes(ctypes.byref(d)))


def qmoe_w4a16_h_to_f16(d, h_tiles, offsets, h16_tiles, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_w4a16_h_to_f16(ctypes.byref(d), _ptr(h_tiles), _ptr(offsets), _ptr(h16_tiles), wp, wn,
                                     _stream(stream)), "qmoe_w4a16_h_to_f16")


def qmoe_permute_x_f16(d, x, sorted_pair_ids, offsets, x_tiles, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_permute_x_f16(ctypes.byref(d), _ptr(x), _ptr(sorted_pair_ids), _ptr(offsets), _ptr(x_tiles),
                                    wp, wn, _stream(stream)), "qmoe_permute_x_f16")


def qmoe_gemm1_swiglu_w4a16(d, x_tiles, w1, offsets, h_tiles, status, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_gemm1_swiglu_w4a16(ctypes.byref(d), _ptr(x_tiles), _ptr(w1), _ptr(offsets), _ptr(h_tiles),
                                         _ptr(status), wp, wn, _stream(stream)), "qmoe_gemm1_swiglu_w4a16")


def mx_tiles_bytes(d: Dims, K: int) -> int:
    return int(lib().qmoe_mx_tiles_bytes(ctypes.byref(d), K))


def qmoe_permute_quant_mxfp8(d, x, pair_slot, offsets, x_tiles, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_permute_quant_mxfp8(ctypes.byref(d), _ptr(x), _ptr(pair_slot), _ptr(offsets),
                                          _ptr(x_tiles), wp, wn, _stream(stream)), "qmoe_permute_quant_mxfp8")


def qmoe_gemm1_swiglu_mxfp4(d, x_tiles, w1, w1_s, offsets, h_tiles, status, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_gemm1_swiglu_mxfp4(ctypes.byref(d), _ptr(x_tiles), _ptr(w1), _ptr(w1_s), _ptr(offsets),
                                         _ptr(h_tiles), _ptr(status), wp, wn, _stream(stream)),
           "qmoe_gemm1_swiglu_mxfp4")


def qmoe_gemm1_swiglu_mxfp4_gather(d, x_q, x_s, sorted_pair_ids, w1, w1_s, offsets, h_tiles, status, ws,
                                   stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_gemm1_swiglu_mxfp4_gather(ctypes.byref(d), _ptr(x_q), _ptr(x_s), _ptr(sorted_pair_ids),
                                                _ptr(w1), _ptr(w1_s), _ptr(offsets), _ptr(h_tiles), _ptr(status),
                                                wp, wn, _stream(stream)),
           "qmoe_gemm1_swiglu_mxfp4_gather")


def forward_launches(d: Dims, scheme: str) -> int:
    return int(lib().qmoe_forward_launches(ctypes.byref(d), SCHEME_ID[scheme]))


def mx_layer_gathers(d: Dims) -> bool:
    return bool(lib().qmoe_mx_layer_gathers(ctypes.byref(d)))


def w8a8_tiles_bytes(d: Dims, K: int) -> int:
    return int(lib().qmoe_w8a8_tiles_bytes(ctypes.byref(d), K))


def qmoe_permute_quant_int8(d, x, sorted_pair_ids, offsets, x_tiles, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_permute_quant_int8(ctypes.byref(d), _ptr(x), _ptr(sorted_pair_ids), _ptr(offsets),
                                         _ptr(x_tiles), wp, wn, _stream(stream)), "qmoe_permute_quant_int8")


def qmoe_quant_tiles_int8_f32(d, h, offsets, h_tiles, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_quant_tiles_int8_f32(ctypes.byref(d), _ptr(h), _ptr(offsets), _ptr(h_tiles), wp, wn,
                                           _stream(stream)), "qmoe_quant_tiles_int8_f32")


def qmoe_gemm1_swiglu_w8a8(d, x_tiles, w1, w1_s, offsets, h, dbg_acc, status, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_gemm1_swiglu_w8a8(ctypes.byref(d), _ptr(x_tiles), _ptr(w1), _ptr(w1_s), _ptr(offsets), _ptr(h),
                                        _ptr(dbg_acc), _ptr(status), wp, wn, _stream(stream)),
           "qmoe_gemm1_swiglu_w8a8")


def qmoe_gemm2_w4a16(d, h16_tiles, w2, offsets, y, status, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_gemm2_w4a16(ctypes.byref(d), _ptr(h16_tiles), _ptr(w2), _ptr(offsets), _ptr(y), _ptr(status),
                                  wp, wn, _stream(stream)), "qmoe_gemm2_w4a16")


def qmoe_gemm2_mxfp4(d, h_tiles, w2, w2_s, offsets, y, status, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_gemm2_mxfp4(ctypes.byref(d), _ptr(h_tiles), _ptr(w2), _ptr(w2_s), _ptr(offsets), _ptr(y),
                                  _ptr(status), wp, wn, _stream(stream)), "qmoe_gemm2_mxfp4")


def qmoe_gemm2_w8a8(d, h_tiles, w2, w2_s, offsets, y, dbg_acc, status, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_gemm2_w8a8(ctypes.byref(d), _ptr(h_tiles), _ptr(w2), _ptr(w2_s), _ptr(offsets), _ptr(y),
                                 _ptr(dbg_acc), _ptr(status), wp, wn, _stream(stream)), "qmoe_gemm2_w8a8")


def qmoe_combine(d, y, topk_w, pair_slot, out, stream=None):
    _check(lib().qmoe_combine(ctypes.byref(d), _ptr(y), _ptr(topk_w), _ptr(pair_slot), _ptr(out), _stream(stream)),
           "qmoe_combine")


def qmoe_gemm1_swiglu_w4a8(d, x_tiles, w1, w1_s, offsets, h, dbg_acc, status, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_gemm1_swiglu_w4a8(ctypes.byref(d), _ptr(x_tiles), _ptr(w1), _ptr(w1_s), _ptr(offsets), _ptr(h),
                                        _ptr(dbg_acc), _ptr(status), wp, wn, _stream(stream)),
           "qmoe_gemm1_swiglu_w4a8")


def qmoe_gemm2_w4a8(d, h_tiles, w2, w2_s, offsets, y, dbg_acc, status, ws, stream=None):
    wp, wn = _ws(ws)
    _check(lib().qmoe_gemm2_w4a8(ctypes.byref(d), _ptr(h_tiles), _ptr(w2), _ptr(w2_s), _ptr(offsets), _ptr(y),
                                 _ptr(dbg_acc), _ptr(status), wp, wn, _stream(stream)), "qmoe_gemm2_w4a8")


def qmoe_moe_forward(scheme, d, x, topk_ids, topk_w, w1, w1_s, w2, w2_s, out, dev_status, ws, stream=None):
    rc = lib().qmoe_moe_forward(SCHEME_ID[scheme], ctypes.byref(d), _ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w1),
                                _ptr(w1_s), _ptr(w2), _ptr(w2_s), _ptr(out), _ptr(dev_status), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "qmoe_moe_forward")


# ------------------------------------------------------------------ conveniences (torch allocation only)

def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte-aligned byte workspace (torch allocations are 512-aligned)."""
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def moe_forward(scheme, x, topk_ids, topk_w, w1, w1_s, w2, w2_s, H=None, I=None, E=None, ws=None, stream=None):
    """Whole layer through qmoe_moe_forward; returns (out bf16-bits [T, H], dev_status)."""
    T, H_ = x.shape
    k = topk_ids.shape[1]
    E_ = w1.shape[0] if E is None else E
    I_ = (w1.shape[1] // 2) if I is None else I
    d = dims(T, k, H_, I_, E_)
    if ws is None:
        ws = alloc_workspace(forward_workspace_bytes(d, scheme), x.device)
    out = torch.empty((T, H_), dtype=torch.int16, device=x.device)
    status = torch.zeros(1, dtype=torch.int32, device=x.device)
    qmoe_moe_forward(scheme, d, x, topk_ids, topk_w, w1, w1_s, w2, w2_s, out, status, ws, stream)
    return out, status
