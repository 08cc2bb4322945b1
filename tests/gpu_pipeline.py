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
    """Weights as the library takes them (MXFP4 weights and scales pre-packed;
    W4A16 codes pre-packed with their scales, scale slots then unused)."""
    t = {key: dev(inp[key]) for key in ("w1", "w1_s", "w2", "w2_s")}
    if w.scheme == "mxfp4":
        t["w1"], t["w1_s"], t["w2"], t["w2_s"] = qb.prepack_mxfp4(t["w1"], t["w1_s"], t["w2"], t["w2_s"], w.H, w.I)
    elif w.scheme == "w4a16":
        t["w1"], t["w2"] = qb.prepack_w4a16(t["w1"], t["w1_s"], t["w2"], t["w2_s"], w.H, w.I)
        t["w1_s"] = t["w2_s"] = None
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
    y = empty((P, H), torch.int16)  # bf16 bits
    res = {}
    if w.scheme == "w4a16":
        xt = empty(qb.w4a16_x_tiles_bytes(d), torch.uint8)
        ht = empty(qb.w4a16_h_tiles_bytes(d), torch.uint8)
        qb.qmoe_permute_x_f16(d, t["x"], sorted_ids, offsets, xt, ws)
        w1, w2 = qb.prepack_w4a16(t["w1"], t["w1_s"], t["w2"], t["w2_s"], H, I)
        qb.qmoe_gemm1_swiglu_w4a16(d, xt, w1, offsets, ht, status, ws)
        h16 = empty(qb.w4a16_h16_tiles_bytes(d), torch.uint8)
        qb.qmoe_w4a16_h_to_f16(d, ht, offsets, h16, ws)
        qb.qmoe_gemm2_w4a16(d, h16, w2, offsets, y, status, ws)
        res.update(bxt=xt, bht=ht, bh16=h16)
    elif w.scheme == "mxfp4":
        xt = empty(qb.mx_tiles_bytes(d, H), torch.uint8)
        ht = empty(qb.mx_tiles_bytes(d, I), torch.uint8)
        qb.qmoe_permute_quant_mxfp8(d, t["x"], slot, offsets, xt, ws)
        w1, w1p, w2, w2p = qb.prepack_mxfp4(t["w1"], t["w1_s"], t["w2"], t["w2_s"], H, I)
        qb.qmoe_gemm1_swiglu_mxfp4(d, xt, w1, w1p, offsets, ht, status, ws)
        qb.qmoe_gemm2_mxfp4(d, ht, w2, w2p, offsets, y, status, ws)
        res.update(xt=xt, ht=ht)
    else:
        xt = empty(qb.w8a8_tiles_bytes(d, H), torch.uint8)
        qb.qmoe_permute_quant_int8(d, t["x"], sorted_ids, offsets, xt, ws)
        h = empty((P, I), torch.float32)
        acc1 = empty((P, 2 * I), torch.int32) if keep else None
        # W8A8 and W4A8 share the integer activation path; only the weights differ
        g1, g2 = (qb.qmoe_gemm1_swiglu_w8a8, qb.qmoe_gemm2_w8a8) if w.scheme == "w8a8" else \
            (qb.qmoe_gemm1_swiglu_w4a8, qb.qmoe_gemm2_w4a8)
        g1(d, xt, t["w1"], t["w1_s"], offsets, h, acc1, status, ws)
        ht = empty(qb.w8a8_tiles_bytes(d, I), torch.uint8)
        qb.qmoe_quant_tiles_int8_f32(d, h, offsets, ht, ws)
        acc2 = empty((P, H), torch.int32) if keep else None
        g2(d, ht, t["w2"], t["w2_s"], offsets, y, acc2, status, ws)
        res.update(ixt=xt, h=h, iht=ht, acc1=acc1, acc2=acc2)
    out = empty((T, H), torch.int16)
    qb.qmoe_combine(d, y, t["topk_w"], slot, out)
    torch.cuda.synchronize()
    r = dict(out=host(out, np.uint16), status=int(status.item()))
    if keep:
        r.update(offsets=host(offsets), sorted_pair_ids=host(sorted_ids), pair_slot=host(slot), y=host(y, np.uint16))
        for key, v in res.items():
            if v is not None:
                r[key] = host(v, np.uint16) if v.dtype == torch.int16 else host(v)
        if w.scheme == "mxfp4":
            nmax = tile_nmax(T, k, E, H, I)
            r["xq"], r["xs"] = unpack_tiles(r.pop("xt"), r["offsets"], nmax, H)
            r["hq"], r["hs"] = unpack_tiles(r.pop("ht"), r["offsets"], nmax, I)
        elif w.scheme == "w4a16":
            nmax = tile_nmax(T, k, E, H, I)
            nt = max_tiles(P, E, nmax)
            r["x_f16"], r["x_fac"] = unpack_w4_x_tiles(r.pop("bxt"), r["offsets"], nmax, H, nt)
            r["h"], r["h_gmax"] = unpack_w4_h_tiles(r.pop("bht"), r["offsets"], nmax, I, nt)
            r["h_f16"], r["h_fac"] = unpack_w4_x_tiles(r.pop("bh16"), r["offsets"], nmax, I, nt)
        else:
            nmax = tile_nmax(T, k, E, H, I)
            nt = max_tiles(P, E, nmax)
            xt, ht = r.pop("ixt"), r.pop("iht")
            r["xq"], r["xs"] = unpack_i8_tiles(xt, r["offsets"], nmax, H, nt)
            r["hq"], r["hs"] = unpack_i8_tiles(ht, r["offsets"], nmax, I, nt)
            r["x_l1"], r["h_l1"] = unpack_i8_l1max(xt, nmax, H, nt), unpack_i8_l1max(ht, nmax, I, nt)
    return r


# ------------------------------------------------------------------ MX activation tile layout (include/qmoe.h)

def tile_nmax(T, k, E, H, I):
    """The token tile the library uses for these dims (its tile table or default rule)."""
    return qb.tile_nmax(qb.dims(T, k, H, I, E))


def tile_schedule(offsets, nmax):
    cnt = np.diff(offsets.astype(np.int64))
    tiles = (cnt + nmax - 1) // nmax
    return np.concatenate([[0], np.cumsum(tiles)]).astype(np.int64)


def _tile_index(offsets, nmax, slots):
    ts = tile_schedule(offsets, nmax)
    e = np.searchsorted(offsets, slots, side="right") - 1
    local = slots - offsets[e]
    return ts[e] + local // nmax, local % nmax


def _layout(nmax, K, t, r):
    """Byte offsets [rows, K] of codes and [rows, K/32] of scales."""
    nsfb = (nmax + 127) // 128
    bb = nmax * 128 + nsfb * 512
    KT = K // 128
    col = np.arange(K)
    kt, cin = col // 128, col % 128
    chunk, byte = cin // 16, cin % 16
    base = (t[:, None] * KT + kt[None, :]) * bb
    code_off = base + r[:, None] * 128 + ((chunk[None, :] ^ (r[:, None] & 7)) << 4) + byte[None, :]
    blk = np.arange(K // 32)
    sbase = (t[:, None] * KT + (blk // 4)[None, :]) * bb
    scale_off = (sbase + nmax * 128 + (r[:, None] // 128) * 512 + 16 * (r[:, None] % 32) +
                 4 * ((r[:, None] % 128) // 32) + (blk % 4)[None, :])
    return code_off, scale_off


def unpack_tiles(buf, offsets, nmax, K):
    """MX activation tiles -> slot-order codes [P_valid, K] and scales [P_valid, K/32]."""
    slots = np.arange(offsets[-1])
    t, r = _tile_index(offsets, nmax, slots)
    co, so = _layout(nmax, K, t, r)
    return buf[co], buf[so]


def pack_tiles(codes, scales, offsets, nmax, K, nbytes):
    """Slot-order codes/scales -> an MX activation tile buffer of nbytes."""
    buf = np.zeros(nbytes, np.uint8)
    slots = np.arange(offsets[-1])
    t, r = _tile_index(offsets, nmax, slots)
    co, so = _layout(nmax, K, t, r)
    buf[co] = codes[:len(slots)]
    buf[so] = scales[:len(slots)]
    return buf


# ------------------------------------------------------------------ W4A16 activation tile layout (include/qmoe.h)

def max_tiles(P, E, nmax):
    return (P + nmax - 1) // nmax + E


def _w4_layout(nmax, K, t, r):
    """Byte offsets [rows, K] of each 16-bit element (low byte)."""
    KT = K // 64
    col = np.arange(K)
    kt, cin = col // 64, col % 64
    chunk, byte = (2 * cin) // 16, (2 * cin) % 16
    base = (t[:, None] * KT + kt[None, :]) * (nmax * 128)
    return base + r[:, None] * 128 + ((chunk[None, :] ^ (r[:, None] & 7)) << 4) + byte[None, :]


def _gather16(buf, off):
    return buf[off].astype(np.uint16) | (buf[off + 1].astype(np.uint16) << 8)


def unpack_w4_x_tiles(buf, offsets, nmax, H, ntiles):
    """W4A16 x (or h16) tiles -> slot-order fp16 bits [P_valid, K] and per-row factors 2^e [P_valid]."""
    slots = np.arange(offsets[-1])
    t, r = _tile_index(offsets, nmax, slots)
    tail = buf[ntiles * (H // 64) * nmax * 128:].view(np.float32)
    return _gather16(buf, _w4_layout(nmax, H, t, r)), tail[t * nmax + r]


def unpack_w4_h_tiles(buf, offsets, nmax, I, ntiles):
    """W4A16 h tiles -> slot-order bf16 bits [P_valid, I] and group maxima [P_valid, I/32]."""
    slots = np.arange(offsets[-1])
    t, r = _tile_index(offsets, nmax, slots)
    tail = buf[ntiles * (I // 64) * nmax * 128:].view(np.float32)
    g = np.arange(I // 32)
    return _gather16(buf, _w4_layout(nmax, I, t, r)), tail[(t * nmax + r)[:, None] * (I // 32) + g[None, :]]


def pack_w4_h_tiles(rows, offsets, nmax, I, nbytes, ntiles):
    """Slot-order bf16 bits [P_valid, I] -> W4A16 h tiles of nbytes (blocks + group-maxima tail)."""
    buf = np.zeros(nbytes, np.uint8)
    slots = np.arange(offsets[-1])
    t, r = _tile_index(offsets, nmax, slots)
    off = _w4_layout(nmax, I, t, r)
    v = rows[:len(slots)].astype(np.uint16)
    buf[off] = (v & 0xFF).astype(np.uint8)
    buf[off + 1] = (v >> 8).astype(np.uint8)
    mag = ((v.astype(np.uint32) & 0x7FFF) << 16).view(np.float32).reshape(len(slots), I // 32, 32).max(axis=2)
    tail = buf[ntiles * (I // 64) * nmax * 128:].view(np.float32)
    tail[(t * nmax + r)[:, None] * (I // 32) + np.arange(I // 32)[None, :]] = mag
    return buf


# ------------------------------------------------------------------ W8A8 activation tile layout (include/qmoe.h)

def unpack_i8_tiles(buf, offsets, nmax, K, ntiles):
    """W8A8 tiles -> slot-order int8 codes [P_valid, K] (stored as exact fp16 values) and scales [P_valid]."""
    slots = np.arange(offsets[-1])
    t, r = _tile_index(offsets, nmax, slots)
    vals = _gather16(buf, _w4_layout(nmax, K, t, r)).view(np.float16).astype(np.float64)
    q = vals.astype(np.int64)
    assert np.array_equal(q, vals) and np.abs(q).max(initial=0) <= 127, "tile values are not int8 codes"
    tail_off = ntiles * (K // 64) * nmax * 128
    tail = buf[tail_off:tail_off + ntiles * nmax * 4].view(np.float32)
    return q.astype(np.int8), tail[t * nmax + r]


def pack_i8_tiles(codes, scales, offsets, nmax, K, nbytes, ntiles):
    """Slot-order int8 codes [P_valid, K] + scales [P_valid] -> a W8A8 tile buffer of nbytes, with the
    per-(112-row half, 128-element step) maxima of sum |code| the layout in include/qmoe.h states."""
    buf = np.zeros(nbytes, np.uint8)
    slots = np.arange(offsets[-1])
    t, r = _tile_index(offsets, nmax, slots)
    off = _w4_layout(nmax, K, t, r)
    v = codes[:len(slots)].astype(np.float16).view(np.uint16)
    buf[off] = (v & 0xFF).astype(np.uint8)
    buf[off + 1] = (v >> 8).astype(np.uint8)
    tail_off = ntiles * (K // 64) * nmax * 128
    tail = buf[tail_off:tail_off + ntiles * nmax * 4].view(np.float32)
    tail[t * nmax + r] = scales[:len(slots)]
    l1 = i8_step_l1max(codes[:len(slots)], t, r, nmax, K, ntiles)
    buf[tail_off + ntiles * nmax * 4:tail_off + ntiles * nmax * 4 + l1.size * 4] = l1.view(np.uint8)
    return buf


def i8_step_l1max(codes, t, r, nmax, K, ntiles):
    """int32 [ntiles * ceil(nmax/112) * K/128]: per (tile, 112-row half, 128-element step), the max over the
    half's rows of sum |code| over the step."""
    halves = (nmax + 111) // 112
    steps = np.abs(codes.astype(np.int64)).reshape(len(codes), K // 128, 128).sum(axis=2)
    out = np.zeros((ntiles * halves, K // 128), np.int64)
    np.maximum.at(out, t * halves + r // 112, steps)
    return out.astype(np.int32).ravel()


def unpack_i8_l1max(buf, nmax, K, ntiles):
    off = ntiles * (K // 64) * nmax * 128 + ntiles * nmax * 4
    n = ntiles * ((nmax + 111) // 112) * (K // 128)
    return buf[off:off + 4 * n].view(np.int32)
