"""Pins for the CPU oracle: each test ties it to something other than itself
(hand-computed format tables, library dtype casts, closed forms, a dense
brute force, invariants of the routed top-k sum)."""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_mixture_experts_moe_gb300 import inputs as gen
from tests import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "format_tables.txt")


def _tables():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, code, val = line.split()
            rows.append((fmt, int(code), float(val)))
    return rows


DECODERS = {
    "int4": oracle.int4_to_double,
    "e2m1": oracle.e2m1_to_double,
    "e8m0": oracle.e8m0_to_double,
    "e4m3": oracle.e4m3_to_double,
}


@pytest.mark.parametrize("fmt,code,val", _tables())
def test_decode_tables(fmt, code, val):
    got = DECODERS[fmt](code)
    if math.isnan(val):
        assert math.isnan(got)
    else:
        assert got == val and math.copysign(1, got) == math.copysign(1, val)


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_to_double(c)
        if np.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], c


def test_fp16_bf16_decode_match_numpy_torch():
    rng = np.random.default_rng(0)
    h = rng.integers(0, 1 << 16, 4000, dtype=np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    for b, r in zip(h, ref):
        got = oracle.fp16_to_double(b)
        assert (math.isnan(got) and math.isnan(r)) or got == r
    bb = rng.integers(0, 1 << 16, 4000, dtype=np.uint16)
    refb = torch.from_numpy(bb.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    for b, r in zip(bb, refb):
        got = oracle.bf16_to_double(b)
        assert (math.isnan(got) and math.isnan(r)) or got == r


def test_e4m3_encode_roundtrip_and_ties():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        v = oracle.e4m3_to_double(c)
        assert oracle.e4m3_from_double(v) == c
    # ties go to the even mantissa
    assert oracle.e4m3_from_double(1.0625) == 0x38  # between 1.0 and 1.125
    assert oracle.e4m3_from_double(1.1875) == 0x3A  # between 1.125 and 1.25
    assert oracle.e4m3_from_double(2.0 ** -10) == 0x00  # half the smallest subnormal
    assert oracle.e4m3_from_double(3 * 2.0 ** -10) == 0x02
    assert oracle.e4m3_from_double(-(2.0 ** -11)) == 0x80  # keeps the sign of zero
    # saturation
    for v, c in [(448.0, 0x7E), (460.0, 0x7E), (500.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE)]:
        assert oracle.e4m3_from_double(v) == c


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.1, 1, 30, 200)])
    v = np.clip(v, -448, 448).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_double(float(a)) for a in v], np.uint8)
    assert np.array_equal(got, ref)


def _nearest_e4m3_bruteforce(a):
    """Exhaustive nearest finite e4m3 (ties to the even code), then clamp."""
    vals = np.array([oracle.e4m3_to_double(c) for c in range(128) if c != 0x7F])
    codes = np.array([c for c in range(128) if c != 0x7F])
    m = abs(a)
    if m >= 448:
        c = 0x7E
    else:
        d = np.abs(vals - m)
        best = np.flatnonzero(d == d.min())
        c = int(codes[best[0]]) if len(best) == 1 else int([codes[b] for b in best if codes[b] % 2 == 0][0])
    return c | (0x80 if np.signbit(a) else 0)


def test_mx_quant_against_bruteforce():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((6, 64)) * np.array([1e-3, 1, 7, 300, 1e4, 1])[:, None]).astype(np.float32)
    v[5, :32] = 0.0  # an all-zero block
    q, s = oracle.mx_quant(v)
    for r in range(v.shape[0]):
        for b in range(2):
            blk = v[r, 32 * b:32 * b + 32].astype(np.float64)
            amax = np.abs(blk).max()
            if amax == 0:
                assert s[r, b] == 127 and not q[r, 32 * b:32 * b + 32].any()
                continue
            X = math.floor(math.log2(amax)) - 8
            assert s[r, b] == X + 127
            for i in range(32):
                assert q[r, 32 * b + i] == _nearest_e4m3_bruteforce(blk[i] / 2.0 ** X)


def test_mx_quant_special_cases():
    # values already on the grid of the block's scale survive unchanged
    grid = np.array([oracle.e4m3_to_double(c) for c in range(0x70, 0x7F)] * 3, np.float64)[:32]
    grid[0] = 448.0  # amax 448 -> X = 2^0 ... floor(log2 448) = 8 -> X = 1
    q, s = oracle.mx_quant(grid.astype(np.float32)[None, :])
    assert s[0, 0] == 127
    assert np.array_equal([oracle.e4m3_to_double(c) for c in q[0]], grid)
    # amax = 448 * 2^j saturates to the 448 code after scaling
    for j in (-5, 0, 3):
        blk = np.zeros(32, np.float32)
        blk[7] = 448.0 * 2.0 ** j
        blk[8] = -448.0 * 2.0 ** j
        q, s = oracle.mx_quant(blk[None, :])
        assert q[0, 7] == 0x7E and q[0, 8] == 0xFE
        assert oracle.e8m0_to_double(s[0, 0]) * 448 == 448.0 * 2.0 ** j


def test_int8_quant_closed_forms():
    v = np.array([[127.0, -63.5, 0.5, 1.5, -127.0, 2.5, 0.0, 64.4]], np.float32)
    q, s = oracle.int8_quant(v)
    assert s[0] == np.float32(1.0)
    assert q.tolist() == [[127, -64, 0, 2, -127, 2, 0, 64]]
    q, s = oracle.int8_quant(np.zeros((1, 16), np.float32))
    assert s[0] == 1.0 and not q.any()
    rng = np.random.default_rng(3)
    v = rng.standard_normal((5, 300)).astype(np.float32)
    q, s = oracle.int8_quant(v)
    assert np.all(np.abs(q) <= 127)
    assert np.all(np.abs(q * s[:, None].astype(np.float64) - v) <= s[:, None] * 0.5 * (1 + 1e-6))
    assert np.all(np.abs(q).max(axis=1) == 127)


def test_align_sort_matches_stable_argsort():
    rng = np.random.default_rng(4)
    for (T, k, E) in [(1, 1, 1), (16, 2, 8), (300, 10, 512), (1000, 8, 7)]:
        ids = gen.routing_uniform(rng, T, max(E, k), k) % E
        r = oracle.align_sort(ids, E)
        flat = ids.reshape(-1)
        order = np.argsort(flat, kind="stable")
        assert np.array_equal(r["sorted_pair_ids"], order)
        cnt = np.bincount(flat, minlength=E)
        assert np.array_equal(r["counts"], cnt)
        assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(cnt)]))
        inv = np.empty_like(order)
        inv[order] = np.arange(order.size)
        assert np.array_equal(r["pair_slot"], inv)
        assert r["invalid"] == 0


def test_align_sort_invalid_ids():
    ids = np.array([[0, 5], [-1, 2], [9, 0]], np.int32)
    r = oracle.align_sort(ids, 6)
    assert r["invalid"] == 2
    assert r["offsets"][-1] == 4
    assert r["pair_slot"][2] == -1 and r["pair_slot"][4] == -1
    assert r["sorted_pair_ids"].tolist() == [0, 5, 3, 1, -1, -1]


def _tiny(scheme, T=12, H=128, E=6, k=2, I=64, seed=5):
    w = gen.custom(f"tiny_{scheme}", scheme, T, H, E, k, I, seed=seed)
    return w, gen.make_all(w)


@pytest.mark.parametrize("scheme", ["w4a16", "mxfp4", "w8a8", "w4a8"])
def test_forward_matches_dense_bruteforce(scheme):
    w, d = _tiny(scheme)
    dims = (w.T, w.k, w.H, w.I, w.E)
    got = oracle.moe_forward(scheme, dims, d)
    ref = bf.moe_dense(scheme, dims, d)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 1e-10, rel


def test_forward_tiny_config_matches_bruteforce():
    w = gen.WORKLOADS["tiny_w4a16"]
    d = gen.make_all(w)
    dims = (w.T, w.k, w.H, w.I, w.E)
    got = oracle.moe_forward("w4a16", dims, d)
    ref = bf.moe_dense("w4a16", dims, d)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-10


@pytest.mark.parametrize("scheme", ["w4a16", "mxfp4"])
def test_topk1_reduces_to_single_mlp(scheme):
    w, d = _tiny(scheme, k=1)
    d["topk_w"] = np.ones_like(d["topk_w"])
    dims = (w.T, w.k, w.H, w.I, w.E)
    out = oracle.moe_forward(scheme, dims, d)
    # one textbook MLP per token: W2 . Q(silu(W1g a) * W1u a) via numpy matmul
    x = bf.bf16_bits_to_f64(d["x"])
    a = bf.mx_values(x.astype(np.float32)) if scheme == "mxfp4" else x
    W1 = bf.dequant_w(scheme, d["w1"], d["w1_s"])
    W2 = bf.dequant_w(scheme, d["w2"], d["w2_s"])
    for t in range(w.T):
        e = d["topk_ids"][t, 0]
        g = W1[e, :w.I] @ a[t]
        u = W1[e, w.I:] @ a[t]
        h = (g / (1 + np.exp(-g)) * u).astype(np.float32)[None, :]
        hq = bf.mx_values(h)[0] if scheme == "mxfp4" else \
            torch.from_numpy(h).to(torch.bfloat16).double().numpy()[0]
        ref = W2[e] @ hq
        assert np.allclose(out[t], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_w8a8_accumulators_exact():
    w, d = _tiny("w8a8")
    dims = (w.T, w.k, w.H, w.I, w.E)
    out, dbg, inv = oracle.moe_forward("w8a8", dims, d, debug=True)
    xq, xs = oracle.quant_act("w8a8", d["x"])
    for t in range(w.T):
        for j in range(w.k):
            e = d["topk_ids"][t, j]
            ref = d["w1"][e].astype(np.int64) @ xq[t].astype(np.int64)
            assert np.array_equal(dbg["acc1"][t * w.k + j], ref)
    # stage-2 accumulators on the quantised intermediate
    experts = d["topk_ids"].reshape(-1)
    y, acc2 = oracle.stage2("w8a8", w.H, w.I, w.E, experts, dbg["hq"], dbg["hs"], d["w2"], d["w2_s"], acc=True)
    for r in range(experts.size):
        ref = d["w2"][experts[r]].astype(np.int64) @ dbg["hq"][r].astype(np.int64)
        assert np.array_equal(acc2[r], ref)
    assert np.array_equal(y, dbg["y"])


def test_w4a8_is_w8a8_on_the_widened_codes():
    # W4A8 reduces to W8A8 once the int4 nibbles are written out as int8 values
    w, d = _tiny("w4a8", seed=19)
    dims = (w.T, w.k, w.H, w.I, w.E)
    out4, dbg4, _ = oracle.moe_forward("w4a8", dims, d, debug=True)
    widen = lambda b: (bf.unpack_nibbles(b).astype(np.int16) - 8).astype(np.int8)
    d8 = dict(d, w1=widen(d["w1"]), w2=widen(d["w2"]))
    assert d8["w1"].min() >= -7 and d8["w1"].max() <= 7
    out8, dbg8, _ = oracle.moe_forward("w8a8", dims, d8, debug=True)
    assert np.array_equal(out4, out8)
    assert np.array_equal(dbg4["acc1"], dbg8["acc1"])
    # the gate/up accumulators are the integer products of the widened codes
    xq, _ = oracle.quant_act("w4a8", d["x"])
    for t in range(w.T):
        for j in range(w.k):
            e = d["topk_ids"][t, j]
            assert np.array_equal(dbg4["acc1"][t * w.k + j], d8["w1"][e].astype(np.int64) @ xq[t].astype(np.int64))


def test_w4a8_largest_sums_fit_fp32_exactly():
    # |code| <= 7 and |x| <= 127: every partial sum of a K <= 16384 dot stays below 2^24
    assert 7 * 127 * 16384 < 2 ** 24
    K = 16384
    a = np.full(K, 127, np.int64)
    w_ = np.full(K, -7, np.int64)
    s = int(a @ w_)
    assert s == -7 * 127 * K and float(np.float32(s)) == s


def test_w8a8_adversarial_extremes_fit_int32():
    # all +-127 operands: the largest |dot| a K=4096 row can reach
    K = 4096
    a = np.full(K, 127, np.int8)
    w_ = np.full(K, -127, np.int8)
    ref = int(a.astype(np.int64) @ w_.astype(np.int64))
    assert ref == -127 * 127 * K and abs(ref) < 2 ** 31


@pytest.mark.parametrize("scheme", ["w4a16", "mxfp4", "w8a8", "w4a8"])
def test_invariants(scheme):
    w, d = _tiny(scheme, seed=11)
    dims = (w.T, w.k, w.H, w.I, w.E)
    base = oracle.moe_forward(scheme, dims, d)
    # permuting tokens permutes the output
    perm = np.random.default_rng(0).permutation(w.T)
    d2 = dict(d, x=d["x"][perm], topk_ids=d["topk_ids"][perm], topk_w=d["topk_w"][perm])
    assert np.array_equal(oracle.moe_forward(scheme, dims, d2), base[perm])
    # relabelling experts (with the weights permuted to match) changes nothing
    lab = np.random.default_rng(1).permutation(w.E)
    inv = np.argsort(lab)
    d3 = dict(d, topk_ids=lab[d["topk_ids"]].astype(np.int32),
              w1=d["w1"][inv], w1_s=d["w1_s"][inv], w2=d["w2"][inv], w2_s=d["w2_s"][inv])
    assert np.array_equal(oracle.moe_forward(scheme, dims, d3), base)
    # scaling the routing weights by 2 scales the output by exactly 2
    d4 = dict(d, topk_w=(d["topk_w"] * 2).astype(np.float32))
    assert np.array_equal(oracle.moe_forward(scheme, dims, d4), 2 * base)
    # x = 0 and W2 = 0 give 0
    d5 = dict(d, x=np.zeros_like(d["x"]))
    assert not oracle.moe_forward(scheme, dims, d5).any()
    zero_w2 = np.zeros_like(d["w2"]) if scheme == "w8a8" else \
        np.full_like(d["w2"], 0x88 if scheme in ("w4a16", "w4a8") else 0)
    d6 = dict(d, w2=zero_w2)
    assert not oracle.moe_forward(scheme, dims, d6).any()
    # a token subset returns exactly those rows
    sub = np.array([3, 0, 7])
    assert np.array_equal(oracle.moe_forward(scheme, dims, d, tokens=sub), base[sub])


@pytest.mark.parametrize("scheme", ["w4a16", "mxfp4"])
def test_stage2_agrees_with_forward_intermediates(scheme):
    w, d = _tiny(scheme, seed=13)
    dims = (w.T, w.k, w.H, w.I, w.E)
    out, dbg, _ = oracle.moe_forward(scheme, dims, d, debug=True)
    experts = d["topk_ids"].reshape(-1)
    y = oracle.stage2(scheme, w.H, w.I, w.E, experts, dbg["hq"], dbg.get("hs"), d["w2"], d["w2_s"])
    assert np.array_equal(y, dbg["y"])
    # and the weighted sum of the y rows, j ascending, is the output
    tw = d["topk_w"].astype(np.float64)
    acc = np.zeros_like(out)
    for j in range(w.k):
        acc += tw[:, j:j + 1] * y.reshape(w.T, w.k, w.H)[:, j]
    assert np.array_equal(acc, out)


def test_invalid_ids_contribute_nothing():
    w, d = _tiny("w4a16", seed=17)
    dims = (w.T, w.k, w.H, w.I, w.E)
    base = oracle.moe_forward("w4a16", dims, d)
    d2 = dict(d, topk_ids=d["topk_ids"].copy())
    d2["topk_ids"][4, 1] = w.E + 3
    out, _, invalid = oracle.moe_forward("w4a16", dims, d2, debug=True)
    assert invalid == 1
    y_removed = base[4] - out[4]
    assert np.abs(y_removed).max() > 0
    others = np.arange(w.T) != 4
    assert np.array_equal(out[others], base[others])


def test_activation_quant_mx_exact_from_bf16():
    # bf16 inputs make the MX decision exact: dequantised codes equal the
    # nearest-e4m3 of x / X for every element
    w, d = _tiny("mxfp4", seed=19)
    q, s = oracle.quant_act("mxfp4", d["x"])
    x = bf.bf16_bits_to_f64(d["x"])
    deq = np.vectorize(oracle.e4m3_to_double)(q) * np.repeat(np.exp2(s.astype(np.float64) - 127), 32, axis=1)
    assert np.array_equal(deq, bf.mx_values(x.astype(np.float32)))


def test_combine_hand_computed():
    # two tokens, top-2, two columns; pair 3 is unrouted (slot -1).  Rows of y
    # are in slot order.  [hip-ep] description: the scatter back is a fixed-order
    # weighted sum over the token's routed pairs.
    y = np.array([[1.0, -2.0], [0.5, 4.0], [3.0, 0.25]], np.float32)
    topk_w = np.array([[0.25, 0.75], [2.0, -1.0]], np.float32)
    pair_slot = np.array([2, 0, 1, -1], np.int32)
    # token 0: 0.25*(3, 0.25) + 0.75*(1, -2) = (1.5, -1.4375)
    # token 1: 2*(0.5, 4); its second pair is skipped
    out = oracle.combine(y, topk_w, pair_slot)
    assert out.tolist() == [[1.5, -1.4375], [1.0, 8.0]]


def test_combine_matches_einsum_over_gathered_rows():
    rng = np.random.default_rng(23)
    T, k, H = 37, 5, 48
    P = T * k
    y = rng.standard_normal((P + 3, H)).astype(np.float32)  # three spare rows nothing points at
    topk_w = rng.uniform(0.05, 1.0, (T, k)).astype(np.float32)
    pair_slot = rng.permutation(P + 3)[:P].astype(np.int32)
    pair_slot[[4, 17, 100]] = -1
    got = oracle.combine(y, topk_w, pair_slot)
    rows = y.astype(np.float64)[np.maximum(pair_slot, 0)].reshape(T, k, H)
    mask = (pair_slot >= 0).reshape(T, k).astype(np.float64)
    ref = np.einsum("tj,tjh->th", topk_w.astype(np.float64) * mask, rows)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("scheme", ["w4a16", "mxfp4", "w8a8"])
def test_combine_of_forward_rows_gives_forward_output(scheme):
    # the forward's own per-pair y rows (pair order, so pair_slot is the
    # identity), rounded to fp32, recombine to its output within that rounding;
    # an unrouted pair removes exactly its weighted row
    w, d = _tiny(scheme, seed=29)
    dims = (w.T, w.k, w.H, w.I, w.E)
    out, dbg, _ = oracle.moe_forward(scheme, dims, d, debug=True)
    y32 = dbg["y"].astype(np.float32)
    P = w.T * w.k
    ident = np.arange(P, dtype=np.int32)
    got = oracle.combine(y32, d["topk_w"], ident)
    bound = (np.abs(d["topk_w"].astype(np.float64))[:, :, None] *
             np.abs(dbg["y"]).reshape(w.T, w.k, w.H)).sum(1) * 2.0 ** -23 + 1e-300
    assert (np.abs(got - out) <= bound).all()
    cut = ident.copy()
    cut[2 * w.k + 1] = -1
    got2 = oracle.combine(y32, d["topk_w"], cut)
    removed = float(d["topk_w"][2, 1]) * y32[2 * w.k + 1].astype(np.float64)
    assert np.allclose(got[2] - got2[2], removed, rtol=1e-12, atol=1e-12 * np.abs(removed).max())
    others = np.arange(w.T) != 2
    assert np.array_equal(got[others], got2[others])
