"""Seeded synthetic inputs for the quantized MoE expert path.

This module holds raw random draws only: routing ids and weights, activation
values, and packed weight/scale bytes drawn directly in their storage formats.
It contains no quantisation, dequantisation, GEMM, activation or combine
arithmetic; the CUDA library and the CPU oracle each implement those on their
own, and both are fed from here.

Workloads follow the shapes the source pages describe:
  * "perf(qmoe): group prefill expert matmuls" -- symmetric int4 expert
    projections (W4A16 here, per-32 fp16 scales).
  * "Evaluate native IU4/IU8 WMMA for grouped-INT MoE prefill on gfx1151",
    Constraint -- int8 x int8 with int32 accumulation (W8A8 here), and int4
    weights widened to 8-bit integers before the integer MMA (W4A8 here:
    int4 codes with per-output-channel fp32 scales, int8 activations).
  * the aiter tuned grouped-fmoe page, Changes -- model_dim 4096, 512 experts,
    top-10, inter_dim 1024, fp8 activations with MXFP4 weights.
The pages measure on real models and GSM8K; none is available here, so every
tensor is a seeded synthetic stand-in with the stated shapes and value
distributions.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

SCHEMES = ("w4a16", "mxfp4", "w8a8", "w4a8")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    scheme: str
    T: int
    H: int
    E: int
    k: int
    I: int
    routing: str  # "uniform" (k distinct experts per token) or "zipf"
    seed: int     # routing and activations
    wseed: int    # expert weights (shared by the members of a T sweep)

    @property
    def P(self) -> int:
        return self.T * self.k

    def flops(self) -> float:
        """Algorithmic flops of one pass: 4*P*H*I (gate+up) + 2*P*H*I (down)."""
        return 6.0 * self.P * self.H * self.I


def _mk(name, scheme, T, H, E, k, I, routing, seed, wseed=None):
    return Workload(name, scheme, T, H, E, k, I, routing, seed, seed if wseed is None else wseed)


# Seeds are 1000 + the workload family index; sweep members add T.
WORKLOADS = {
    w.name: w
    for w in [
        _mk("tiny_w4a16", "w4a16", 16, 256, 8, 2, 128, "uniform", 1000),
        _mk("w4a16_T2048", "w4a16", 2048, 2048, 128, 8, 768, "uniform", 1001),
        *[
            _mk(f"mxfp4_T{T}", "mxfp4", T, 4096, 512, 10, 1024, "uniform", 1002 + T, 1002)
            for T in (256, 1024, 4096, 8192)
        ],
        _mk("w8a8_T8192", "w8a8", 8192, 4096, 64, 8, 1408, "uniform", 1003),
        # int4 weights widened to 8-bit integers, int8 activations: the W8A8 layer's shape
        _mk("w4a8_T8192", "w4a8", 8192, 4096, 64, 8, 1408, "uniform", 1010),
        *[
            _mk(f"decode_T{T}", "mxfp4", T, 4096, 512, 10, 1024, "zipf", 1004 + T, 1002)
            for T in (1, 4, 16, 64)
        ],
        # tensor-parallel shards of the MXFP4 layer: TP2 keeps inter 512 of
        # the 1024 columns per rank, TP4 keeps 256 (same experts, hidden, top-k)
        *[
            _mk(f"mxfp4_tp{tp}_T{T}", "mxfp4", T, 4096, 512, 10, 1024 // tp, "uniform", 1005 + tp + T, 1005 + tp)
            for tp in (2, 4)
            for T in (16, 256, 1024, 4096, 8192)
        ],
        # profiling stand-in for the T=4096 MXFP4 layer: same per-expert load
        # (about 80 tokens), 64 experts so a capture holds ~0.5 GB of weights
        _mk("prof_mxfp4_E64_T512", "mxfp4", 512, 4096, 64, 10, 1024, "uniform", 1005),
        # profiling stand-in for the gathering stage 1 of the TP4 shard (I 256) at T=4096: same
        # per-expert load (about 80 tokens), 128 experts (~0.14 GB of stage-1 weights, above L2)
        _mk("prof_mxfp4_tp4_E128_T1024", "mxfp4", 1024, 4096, 128, 10, 256, "uniform", 1012),
        # profiling stand-in for the routing sort, permute and combine of the T=4096 MXFP4
        # layer: the same 4096 tokens and 40960 pairs, 16 experts (~70 MB of weights)
        _mk("prof_small_E16_T4096", "mxfp4", 4096, 4096, 16, 10, 1024, "uniform", 1008),
        # profiling stand-in for the T=8192 W8A8 layer: same per-expert load
        # (about 1024 tokens), 8 experts (~0.14 GB of weights)
        _mk("prof_w8a8_E8_T1024", "w8a8", 1024, 4096, 8, 8, 1408, "uniform", 1006),
        # the same stand-in for the W4A8 layer
        _mk("prof_w4a8_E8_T1024", "w4a8", 1024, 4096, 8, 8, 1408, "uniform", 1011),
    ]
}


def custom(name, scheme, T, H, E, k, I, routing="uniform", seed=7):
    """A workload outside the fixed table (small parity and edge cases)."""
    return Workload(name, scheme, T, H, E, k, I, routing, seed, seed)


def rng_for(w: Workload, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([w.seed, stream]))


def _raw_bytes(rng: np.random.Generator, n: int) -> np.ndarray:
    """n uniform random bytes (fast path: raw 64-bit PCG64 output)."""
    words = rng.bit_generator.random_raw((n + 7) // 8)
    return words.view(np.uint8)[:n].copy()


def bf16_bits_from_f32(v: np.ndarray) -> np.ndarray:
    """Storage conversion of a float32 draw to bfloat16 bits (round to nearest even)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


# ---------------------------------------------------------------- routing


def routing_uniform(rng, T, E, k):
    """k distinct experts per token, uniform over the E experts."""
    keys = rng.random((T, E))
    ids = np.argsort(keys, axis=1, kind="stable")[:, :k]
    return ids.astype(np.int32)


def routing_zipf(rng, T, E, k, s=1.2):
    """k distinct experts per token, skewed: experts are ranked by a seeded
    permutation and drawn without replacement with probability ~ rank^-s
    (Gumbel-top-k over logits -s*ln(rank))."""
    rank_of = rng.permutation(E)  # rank_of[e] in 0..E-1
    logits = -s * np.log(rank_of.astype(np.float64) + 1.0)
    g = rng.gumbel(size=(T, E))
    ids = np.argsort(-(logits[None, :] + g), axis=1, kind="stable")[:, :k]
    return ids.astype(np.int32)


def routing_weights(rng, T, k):
    """Softmax of N(0,1) logits over the k chosen experts, as float32."""
    z = rng.standard_normal((T, k))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


def routing_with_counts(rng, counts, k):
    """Routing whose per-expert load is exactly `counts` (sum = T*k), with
    each token's k experts distinct.  Used for ragged-tail cases such as
    expert loads of 0, 1, 127 and 129 pairs."""
    counts = np.asarray(counts, dtype=np.int64)
    E = len(counts)
    P = int(counts.sum())
    assert P % k == 0
    T = P // k
    # Round-robin the pair list sorted by expert into k columns: consecutive
    # pairs of the sorted list land in different tokens, so as long as no
    # expert holds more than T pairs, every token's k experts are distinct.
    assert counts.max() <= T
    flat = np.repeat(np.arange(E, dtype=np.int32), counts)
    ids = flat.reshape(k, T).T.copy()
    perm = rng.permutation(T)
    return ids[perm].astype(np.int32)


# ---------------------------------------------------------------- weights


def int4_bytes(rng, shape_bytes):
    """Packed symmetric int4: each byte holds two independent nibbles, each
    uniform over 1..15 (stored n = q + 8, q uniform in [-7, 7])."""
    lo = rng.integers(1, 16, size=shape_bytes, dtype=np.uint8)
    hi = rng.integers(1, 16, size=shape_bytes, dtype=np.uint8)
    return (lo | (hi << 4)).astype(np.uint8)


def fp16_scales(rng, shape, lo=0.005, hi=0.02):
    return rng.uniform(lo, hi, size=shape).astype(np.float16)


def e2m1_bytes(rng, shape_bytes):
    """Packed E2M1: two independent codes per byte, uniform over all 16 codes."""
    n = int(np.prod(shape_bytes))
    return _raw_bytes(rng, n).reshape(shape_bytes)


def e8m0_bytes(rng, shape, lo=119, hi=123):
    """E8M0 scale bytes uniform over [lo, hi] (2^-8 .. 2^-4 by default)."""
    return rng.integers(lo, hi + 1, size=shape, dtype=np.uint8)


def int8_values(rng, shape):
    return rng.integers(-127, 128, size=shape, dtype=np.int8)


def int8_channel_scales(rng, shape, K, qmax=127.0):
    """Per-output-channel fp32 scales U(0.5, 1.5) / (qmax * sqrt(K))."""
    return (rng.uniform(0.5, 1.5, size=shape) / (qmax * math.sqrt(K))).astype(np.float32)


# ---------------------------------------------------------------- bundles


def make_routing(w: Workload):
    rng = rng_for(w, 1)
    if w.routing == "zipf":
        ids = routing_zipf(rng, w.T, w.E, w.k)
    else:
        ids = routing_uniform(rng, w.T, w.E, w.k)
    return ids, routing_weights(rng, w.T, w.k)


def make_activations(w: Workload):
    """bf16 activations drawn from N(0,1) (uint16 bit patterns, [T, H])."""
    rng = rng_for(w, 2)
    return bf16_bits_from_f32(rng.standard_normal((w.T, w.H), dtype=np.float32))


def make_weights(w: Workload):
    """Expert weights in storage format.

    W1 is [E, 2I, H] (rows 0..I-1 gate, I..2I-1 up), W2 is [E, H, I]; K is the
    last (contiguous) axis in both.  Packed 4-bit formats hold K/2 bytes/row."""
    rng = np.random.Generator(np.random.PCG64([w.wseed, 3]))
    E, H, I = w.E, w.H, w.I
    if w.scheme == "w4a16":
        return dict(
            w1=int4_bytes(rng, (E, 2 * I, H // 2)),
            w1_s=fp16_scales(rng, (E, 2 * I, H // 32)),
            w2=int4_bytes(rng, (E, H, I // 2)),
            w2_s=fp16_scales(rng, (E, H, I // 32)),
        )
    if w.scheme == "mxfp4":
        return dict(
            w1=e2m1_bytes(rng, (E, 2 * I, H // 2)),
            w1_s=e8m0_bytes(rng, (E, 2 * I, H // 32)),
            w2=e2m1_bytes(rng, (E, H, I // 2)),
            w2_s=e8m0_bytes(rng, (E, H, I // 32)),
        )
    if w.scheme == "w8a8":
        return dict(
            w1=int8_values(rng, (E, 2 * I, H)),
            w1_s=int8_channel_scales(rng, (E, 2 * I), H),
            w2=int8_values(rng, (E, H, I)),
            w2_s=int8_channel_scales(rng, (E, H), I),
        )
    if w.scheme == "w4a8":
        return dict(
            w1=int4_bytes(rng, (E, 2 * I, H // 2)),
            w1_s=int8_channel_scales(rng, (E, 2 * I), H, 7.0),
            w2=int4_bytes(rng, (E, H, I // 2)),
            w2_s=int8_channel_scales(rng, (E, H), I, 7.0),
        )
    raise ValueError(w.scheme)


def make_all(w: Workload, routing=None):
    ids, tw = make_routing(w) if routing is None else routing
    d = dict(x=make_activations(w), topk_ids=ids, topk_w=tw)
    d.update(make_weights(w))
    return d


def make_stage2_inputs(w: Workload, rows: int):
    """Random already-quantised intermediate rows for testing the down
    projection on its own: one expert id per row (sorted) plus the row's codes."""
    rng = rng_for(w, 4)
    experts = np.sort(rng.integers(0, w.E, size=rows)).astype(np.int32)
    I = w.I
    if w.scheme == "w4a16":
        h = bf16_bits_from_f32(rng.standard_normal((rows, I), dtype=np.float32))
        return dict(experts=experts, h=h)
    if w.scheme == "mxfp4":
        codes = _raw_bytes(rng, rows * I).reshape(rows, I)
        codes[(codes & 0x7F) == 0x7F] ^= 0x01  # no NaN codes: 0x7F/0xFF -> 0x7E/0xFE
        return dict(experts=experts, h=codes, h_s=e8m0_bytes(rng, (rows, I // 32), 118, 126))
    if w.scheme in ("w8a8", "w4a8"):
        return dict(
            experts=experts,
            h=int8_values(rng, (rows, I)),
            h_s=rng.uniform(0.001, 0.05, size=rows).astype(np.float32),
        )
    raise ValueError(w.scheme)
