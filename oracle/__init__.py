"""CPU oracle for the quantized MoE expert path -- TEST INFRASTRUCTURE.

Only tests/, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its binding) never
imports it and fails loudly when the CUDA library is missing.

The arithmetic lives in qmoe_oracle.c (plain C, double accumulation, OpenMP
over tokens); this module builds it with gcc and marshals numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmoe_oracle.c")
_LIB = os.path.join(_HERE, "libqmoe_oracle.so")

SCHEME_ID = {"w4a16": 0, "mxfp4": 1, "w8a8": 2, "w4a8": 3}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = [
        "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
        "-ffp-contract=off", "-fno-fast-math", "-Wall",
        _SRC, "-o", tmp, "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        # A planted-mistake test points this at a mutated build of the oracle.
        path = os.environ.get("QMOE_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        d, u8, u16, i64, i32, vp = (
            ctypes.c_double, ctypes.c_uint8, ctypes.c_uint16, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p)
        for name in ("oracle_bf16_to_double", "oracle_fp16_to_double"):
            getattr(L, name).argtypes = [u16]
            getattr(L, name).restype = d
        for name in ("oracle_int4_to_double", "oracle_e2m1_to_double", "oracle_e8m0_to_double",
                     "oracle_e4m3_to_double"):
            getattr(L, name).argtypes = [u8]
            getattr(L, name).restype = d
        L.oracle_e4m3_from_double_sat.argtypes = [d]
        L.oracle_e4m3_from_double_sat.restype = u8
        L.oracle_float_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_float_to_bf16.restype = u16
        L.oracle_mx_quant.argtypes = [vp, i64, vp, vp]
        L.oracle_mx_quant.restype = None
        L.oracle_int8_quant.argtypes = [vp, i64, i64, vp, vp]
        L.oracle_int8_quant.restype = None
        L.oracle_quant_act.argtypes = [i32, i64, i64, vp, vp, vp]
        L.oracle_quant_act.restype = i32
        L.oracle_align_sort.argtypes = [i64, i32, vp, vp, vp, vp, vp]
        L.oracle_align_sort.restype = i64
        L.oracle_stage2.argtypes = [i32, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        L.oracle_stage2.restype = i32
        L.oracle_moe_forward.argtypes = [i32, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, i64, vp, vp,
                                         vp, vp, vp, vp, vp]
        L.oracle_moe_forward.restype = i64
        L.oracle_combine.argtypes = [i64, i32, i32, vp, vp, vp, vp]
        L.oracle_combine.restype = None
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = i32
        _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------ scalar formats

def bf16_to_double(b): return lib().oracle_bf16_to_double(int(b))
def fp16_to_double(b): return lib().oracle_fp16_to_double(int(b))
def int4_to_double(n): return lib().oracle_int4_to_double(int(n))
def e2m1_to_double(c): return lib().oracle_e2m1_to_double(int(c))
def e8m0_to_double(b): return lib().oracle_e8m0_to_double(int(b))
def e4m3_to_double(b): return lib().oracle_e4m3_to_double(int(b))
def e4m3_from_double(v): return lib().oracle_e4m3_from_double_sat(float(v))
def float_to_bf16(v): return lib().oracle_float_to_bf16(float(v))


def num_threads() -> int:
    return lib().oracle_num_threads()


# ------------------------------------------------------------ quantisers

def mx_quant(v: np.ndarray):
    """MX (e4m3 + E8M0 per 32) quantisation of fp32 rows [..., n]."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    q = np.empty(v.shape, np.uint8)
    s = np.empty(v.shape[:-1] + (v.shape[-1] // 32,), np.uint8)
    lib().oracle_mx_quant(_p(v), v.size, _p(q), _p(s))
    return q, s


def int8_quant(v: np.ndarray):
    """Per-row int8 quantisation of fp32 rows [rows, n]."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    rows, n = v.shape
    q = np.empty(v.shape, np.int8)
    s = np.empty(rows, np.float32)
    lib().oracle_int8_quant(_p(v), rows, n, _p(q), _p(s))
    return q, s


def quant_act(scheme: str, x_bf16: np.ndarray):
    """The scheme's activation quantisation of bf16 rows [rows, cols]."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, cols = x.shape
    if scheme == "mxfp4":
        q = np.empty((rows, cols), np.uint8)
        s = np.empty((rows, cols // 32), np.uint8)
    elif scheme in ("w8a8", "w4a8"):
        q = np.empty((rows, cols), np.int8)
        s = np.empty(rows, np.float32)
    else:
        raise ValueError(scheme)
    rc = lib().oracle_quant_act(SCHEME_ID[scheme], rows, cols, _p(x), _p(q), _p(s))
    assert rc == 0
    return q, s


# ------------------------------------------------------------ routing

def align_sort(topk_ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32).reshape(-1)
    P = ids.size
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    sorted_ids = np.empty(P, np.int32)
    pair_slot = np.empty(P, np.int32)
    invalid = lib().oracle_align_sort(P, E, _p(ids), _p(counts), _p(offsets), _p(sorted_ids), _p(pair_slot))
    return dict(counts=counts, offsets=offsets, sorted_pair_ids=sorted_ids, pair_slot=pair_slot,
                invalid=int(invalid))


# ------------------------------------------------------------ MoE

def moe_forward(scheme: str, dims, inp: dict, tokens=None, debug: bool = False):
    """Full forward.  dims = (T, k, H, I, E); inp holds x, topk_ids, topk_w,
    w1, w1_s, w2, w2_s as produced by the input generator.  `tokens` selects
    a subset of tokens (rows of the result follow that order)."""
    T, k, H, I, E = dims
    if tokens is None:
        ntok, tl = T, None
    else:
        tl = np.ascontiguousarray(tokens, dtype=np.int64)
        ntok = tl.size
    out = np.zeros((ntok, H), np.float64)
    R = ntok * k
    dbg = {}
    if debug:
        dbg["h"] = np.zeros((R, I), np.float32)
        if scheme == "w4a16":
            dbg["hq"] = np.zeros((R, I), np.uint16)
        elif scheme == "mxfp4":
            dbg["hq"] = np.zeros((R, I), np.uint8)
            dbg["hs"] = np.zeros((R, I // 32), np.uint8)
        else:
            dbg["hq"] = np.zeros((R, I), np.int8)
            dbg["hs"] = np.zeros(R, np.float32)
            dbg["acc1"] = np.zeros((R, 2 * I), np.int32)
        dbg["y"] = np.zeros((R, H), np.float64)
    c = lambda a: np.ascontiguousarray(a)
    rc = lib().oracle_moe_forward(
        SCHEME_ID[scheme], T, k, H, I, E, _p(c(inp["x"])), _p(c(inp["topk_ids"])), _p(c(inp["topk_w"])),
        _p(c(inp["w1"])), _p(c(inp["w1_s"])), _p(c(inp["w2"])), _p(c(inp["w2_s"])), ntok, _p(tl), _p(out),
        _p(dbg.get("h")), _p(dbg.get("hq")), _p(dbg.get("hs")), _p(dbg.get("acc1")), _p(dbg.get("y")))
    if rc == -(1 << 30):
        raise OverflowError("an integer dot product does not fit int32")
    if debug:
        return out, dbg, -int(rc)
    return out


def stage2(scheme: str, H: int, I: int, E: int, experts, h, h_s, w2, w2_s, acc: bool = False):
    """Down projection of already-quantised rows (row r through experts[r])."""
    experts = np.ascontiguousarray(experts, dtype=np.int32)
    rows = experts.size
    y = np.zeros((rows, H), np.float64)
    acc2 = np.zeros((rows, H), np.int32) if acc else None
    c = lambda a: None if a is None else np.ascontiguousarray(a)
    rc = lib().oracle_stage2(SCHEME_ID[scheme], rows, H, I, E, _p(experts), _p(c(h)), _p(c(h_s)), _p(c(w2)),
                             _p(c(w2_s)), _p(y), _p(acc2))
    if rc != 0:
        raise RuntimeError(f"oracle_stage2 failed: {rc}")
    return (y, acc2) if acc else y


def combine(y: np.ndarray, topk_w: np.ndarray, pair_slot: np.ndarray):
    """Top-k weighted sum of fp32 rows y[slot] (j ascending, double)."""
    T, k = topk_w.shape
    H = y.shape[1]
    out = np.zeros((T, H), np.float64)
    c = lambda a, dt: np.ascontiguousarray(a, dtype=dt)
    lib().oracle_combine(T, k, H, _p(c(y, np.float32)), _p(c(topk_w, np.float32)), _p(c(pair_slot, np.int32)),
                         _p(out))
    return out
