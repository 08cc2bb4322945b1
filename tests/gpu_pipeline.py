"""Runs the CUDA path stage by stage through the C ABI (via the ctypes
binding) on numpy inputs from the seeded generator, returning numpy arrays."""

import numpy as np
import torch

from quantized_mixture_experts_moe_gb300 import binding as qb

DEV = "cuda"


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def host(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def empty(shape, dtype):
    return torch.empty(shape, dtype=dtype, device=DEV)


def align(ids: np.ndarray, E: int, T: int, k: int, H=32, I=32):
    d = qb.dims(T, k, H, I, E)
    P = T * k
    t_ids = dev(ids.astype(np.int32).reshape(T, k)) if P else empty((0,), torch.int32)
    counts, offsets = empty(E, torch.int32), empty(E + 1, torch.int32)
    sorted_ids, slot = empty(max(P, 1), torch.int32), empty(max(P, 1), torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = qb.alloc_workspace(qb.workspace_bytes(d))
    qb.qmoe_align_sort(d, t_ids if P else None, counts, offsets, sorted_ids if P else None, slot if P else None,
                       status, ws)
    torch.cuda.synchronize()
    return dict(counts=host(counts), offsets=host(offsets), sorted_pair_ids=host(sorted_ids)[:P],
                pair_slot=host(slot)[:P], status=int(status.item()))


def device_weights(w, inp):
    """Weights as the library takes them (MXFP4 scales pre-packed)."""
    t = {key: dev(inp[key]) for key in ("w1", "w1_s", "w2", "w2_s")}
    if w.scheme == "mxfp4":
        t["w1"], t["w1_s"], t["w2"], t["w2_s"] = qb.prepack_mxfp4(t["w1"], t["w1_s"], t["w2"], t["w2_s"], w.H, w.I)
    return t


def run_layer(w, inp, keep=False):
    """The whole path, one call per stage; returns out (bf16 bits) and, with
    keep=True, every intermediate."""
    T, k, H, I, E = w.T, w.k, w.H, w.I, w.E
    P = T * k
    d = qb.dims(T, k, H, I, E)
    t = {key: dev(v) for key, v in inp.items()}
    counts, offsets = empty(E, torch.int32), empty(E + 1, torch.int32)
    sorted_ids, slot = empty(P, torch.int32), empty(P, torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = qb.alloc_workspace(qb.workspace_bytes(d))
    qb.qmoe_align_sort(d, t["topk_ids"], counts, offsets, sorted_ids, slot, status, ws)
    y = empty((P, H), torch.float32)
    res = {}
    if w.scheme == "w4a16":
        h = empty((P, I), torch.int16)
        qb.qmoe_gemm1_swiglu_w4a16(d, t["x"], t["w1"], t["w1_s"], offsets, sorted_ids, h, status, ws)
        qb.qmoe_gemm2_w4a16(d, h, t["w2"], t["w2_s"], offsets, y, status, ws)
        res["h"] = h
    elif w.scheme == "mxfp4":
        xq, xs = empty((T, H), torch.uint8), empty((T, H // 32), torch.uint8)
        qb.qmoe_quant_act_mxfp8(t["x"], xq, xs)
        hq, hs = empty((P, I), torch.uint8), empty((P, I // 32), torch.uint8)
        w1, w1p, w2, w2p = qb.prepack_mxfp4(t["w1"], t["w1_s"], t["w2"], t["w2_s"], H, I)
        qb.qmoe_gemm1_swiglu_mxfp4(d, xq, xs, w1, w1p, offsets, sorted_ids, hq, hs, status, ws)
        qb.qmoe_gemm2_mxfp4(d, hq, hs, w2, w2p, offsets, y, status, ws)
        res.update(xq=xq, xs=xs, hq=hq, hs=hs)
    else:
        xq, xs = empty((T, H), torch.int8), empty(T, torch.float32)
        qb.qmoe_quant_rows_int8_bf16(t["x"], xq, xs)
        h = empty((P, I), torch.float32)
        acc1 = empty((P, 2 * I), torch.int32) if keep else None
        qb.qmoe_gemm1_swiglu_w8a8(d, xq, xs, t["w1"], t["w1_s"], offsets, sorted_ids, h, acc1, status, ws)
        hq, hs = empty((P, I), torch.int8), empty(P, torch.float32)
        qb.qmoe_quant_rows_int8_f32(h, hq, hs)
        acc2 = empty((P, H), torch.int32) if keep else None
        qb.qmoe_gemm2_w8a8(d, hq, hs, t["w2"], t["w2_s"], offsets, y, acc2, status, ws)
        res.update(xq=xq, xs=xs, h=h, hq=hq, hs=hs, acc1=acc1, acc2=acc2)
    out = empty((T, H), torch.int16)
    qb.qmoe_combine(d, y, t["topk_w"], slot, out)
    torch.cuda.synchronize()
    r = dict(out=host(out, np.uint16), status=int(status.item()))
    if keep:
        r.update(offsets=host(offsets), sorted_pair_ids=host(sorted_ids), pair_slot=host(slot), y=host(y))
        for key, v in res.items():
            if v is not None:
                r[key] = host(v, np.uint16) if v.dtype == torch.int16 else host(v)
    return r
