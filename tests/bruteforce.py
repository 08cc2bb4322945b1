"""Dense masked brute force of the quantized MoE layer (numpy, float64).

An independent formulation used to pin the oracle on tiny inputs: every
token runs through every expert, and the results are summed with the routing
weight of that expert (zero where the token did not pick it).  Decoding uses
lookup tables written from the format definitions; rounding to e4m3 and bf16
uses torch's dtype casts (library routines); nothing is shared with the
oracle's C code.
"""

import numpy as np
import torch

E2M1_TABLE = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], np.float64)


def unpack_nibbles(b: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] nibbles (even K from the low nibble)."""
    lo = b & 0x0F
    hi = b >> 4
    return np.stack([lo, hi], axis=-1).reshape(*b.shape[:-1], b.shape[-1] * 2)


def dequant_w(scheme, w, ws):
    if scheme == "w4a16":
        q = unpack_nibbles(w).astype(np.float64) - 8.0
        s = np.repeat(ws.astype(np.float64), 32, axis=-1)
        return q * s
    if scheme == "mxfp4":
        v = E2M1_TABLE[unpack_nibbles(w)]
        s = np.repeat(np.exp2(ws.astype(np.float64) - 127.0), 32, axis=-1)
        return v * s
    raise ValueError(scheme)


def bf16_bits_to_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_e4m3_values(v: np.ndarray) -> np.ndarray:
    """Nearest e4m3 value (torch cast), after clamping to the finite range."""
    t = torch.from_numpy(np.clip(v, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def mx_values(v32: np.ndarray) -> np.ndarray:
    """MX quantise-dequantise of fp32 rows [..., n] (blocks of 32)."""
    v = v32.astype(np.float64).reshape(*v32.shape[:-1], -1, 32)
    amax = np.abs(v).max(axis=-1, keepdims=True)
    _, ex = np.frexp(amax)
    X = np.clip(ex.astype(np.float64) - 1.0 - 8.0, -127, 127)
    scale = np.exp2(X)
    q = to_e4m3_values(v / scale) * scale
    q = np.where(amax == 0, 0.0, q)
    return q.reshape(v32.shape)


def int8_rows(v32: np.ndarray):
    v32 = v32.astype(np.float32)
    amax = np.abs(v32).max(axis=-1, keepdims=True)
    s = np.where(amax == 0, np.float32(1.0), amax / np.float32(127.0)).astype(np.float32)
    q = np.clip(np.rint(v32 / s), -127, 127).astype(np.int64)
    return q, s[..., 0]


def moe_dense(scheme, dims, inp):
    T, k, H, I, E = dims
    x = bf16_bits_to_f64(inp["x"])  # [T, H]
    ids, tw = inp["topk_ids"], inp["topk_w"].astype(np.float64)
    mask = np.zeros((T, E), np.float64)
    for t in range(T):
        for j in range(k):
            mask[t, ids[t, j]] += tw[t, j]
    out = np.zeros((T, H), np.float64)
    if scheme in ("w8a8", "w4a8"):
        # W4A8: int4 codes widened to integers (nibble n -> n - 8), then the W8A8 arithmetic
        ints = (lambda w: w.astype(np.int64)) if scheme == "w8a8" else \
            (lambda w: unpack_nibbles(w).astype(np.int64) - 8)
        xq, xs = int8_rows(x.astype(np.float32))
        for e in range(E):
            w1 = ints(inp["w1"][e])  # [2I, H]
            acc = xq @ w1.T  # exact integers
            sw = inp["w1_s"][e]
            gu = (acc.astype(np.float32) * xs[:, None]).astype(np.float32) * sw[None, :]
            g, u = gu[:, :I].astype(np.float64), gu[:, I:].astype(np.float64)
            h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
            hq, hs = int8_rows(h)
            acc2 = hq @ ints(inp["w2"][e]).T
            y = (acc2.astype(np.float32) * hs[:, None]).astype(np.float32) * inp["w2_s"][e][None, :]
            out += mask[:, e:e + 1] * y.astype(np.float64)
        return out
    if scheme == "mxfp4":
        a = mx_values(x.astype(np.float32))
    else:
        a = x
    W1 = dequant_w(scheme, inp["w1"], inp["w1_s"])  # [E, 2I, H]
    W2 = dequant_w(scheme, inp["w2"], inp["w2_s"])  # [E, H, I]
    for e in range(E):
        gu = a @ W1[e].T
        g, u = gu[:, :I], gu[:, I:]
        h32 = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
        if scheme == "mxfp4":
            hq = mx_values(h32)
        else:
            hq = torch.from_numpy(h32).to(torch.bfloat16).to(torch.float64).numpy()
        out += mask[:, e:e + 1] * (hq @ W2[e].T)
    return out
