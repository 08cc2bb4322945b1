"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: the permutation, offsets, activation quantisation codes, W8A8
int32 accumulators (and the W8A8 down projection, whose fp32 dequantisation
follows the same operation order on both sides).  Float outputs: relative L2
below 5e-3 (rel L2 = ||gpu - oracle|| / ||oracle|| over all elements,
computed in float64).  Intermediate quantisation codes are compared through
their dequantised values plus a mismatch-rate bound, because fp32 and double
intermediates may straddle a rounding boundary.
"""

import os

import numpy as np
import pytest
import torch

import oracle
from quantized_mixture_experts_moe_gb300 import binding as qb
from quantized_mixture_experts_moe_gb300 import inputs as gen
from tests import bruteforce as bf
from tests import gpu_pipeline as gp

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3
# W4A16 h after stage 1: the weights are single fp16 roundings (<= 2^-11
# relative, ~2e-4 RMS), the activations exact, the sums fp32, so gate/up sit
# ~2e-4 from the oracle's; h's own bf16 rounding (ulp 2^-8 relative) then
# lands on the neighbouring bf16 value for roughly one element in six, which
# a CPU model of this arithmetic puts at rel L2 ~1.0e-3 against the oracle's
# rounded h.  Bound: 2e-3.
W4_H_REL_L2 = 2e-3
# one stage's bf16 y against the double oracle: the bf16 rounding of y is
# ~1.1e-3 rel L2 by itself; 2e-3 leaves room for the fp32 sums and the fp16
# weight rounding (W4A16) without hiding a stage-2 defect twice that size
Y_BF16_REL_L2 = 2e-3


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / (den if den > 0 else 1.0)


def dims(w):
    return (w.T, w.k, w.H, w.I, w.E)


# ------------------------------------------------------------------ routing

ROUTINGS = [
    ("uniform_small", lambda r: gen.routing_uniform(r, 16, 8, 2), 8),
    ("uniform_c3", lambda r: gen.routing_uniform(r, 4096, 512, 10), 512),
    ("zipf_decode", lambda r: gen.routing_zipf(r, 64, 512, 10), 512),
    ("single_token", lambda r: gen.routing_uniform(r, 1, 512, 10), 512),
    ("ragged_loads", lambda r: gen.routing_with_counts(r, [0, 1, 127, 129, 0, 3], 2), 6),
    ("many_chunks", lambda r: gen.routing_uniform(r, 8192, 64, 8), 64),
    ("one_expert_hot", lambda r: np.zeros((5000, 1), np.int32), 4),
]


@pytest.mark.parametrize("name,make,E", ROUTINGS, ids=[r[0] for r in ROUTINGS])
def test_align_sort_bit_exact(name, make, E):
    ids = make(np.random.default_rng(42))
    T, k = ids.shape
    got = gp.align(ids, E, T, k)
    ref = oracle.align_sort(ids, E)
    for key in ("counts", "offsets", "sorted_pair_ids", "pair_slot"):
        assert np.array_equal(got[key], ref[key]), key
    assert got["status"] == 0


def test_align_sort_invalid_ids_set_status():
    ids = np.array([[0, 5], [-1, 2], [9, 0], [3, 3]], np.int32)
    got = gp.align(ids, 6, 4, 2)
    ref = oracle.align_sort(ids, 6)
    assert got["status"] & qb.DEV_BAD_EXPERT_ID
    for key in ("counts", "offsets", "sorted_pair_ids", "pair_slot"):
        assert np.array_equal(got[key], ref[key]), key


def test_align_sort_empty():
    got = gp.align(np.zeros((0, 4), np.int32), 16, 0, 4)
    assert not got["counts"].any() and not got["offsets"].any()


def test_align_sort_deterministic():
    ids = gen.routing_uniform(np.random.default_rng(3), 4096, 512, 10)
    a = gp.align(ids, 512, 4096, 10)
    b = gp.align(ids, 512, 4096, 10)
    assert all(np.array_equal(a[key], b[key]) for key in ("sorted_pair_ids", "pair_slot"))


# ------------------------------------------------------------------ activation quantisation

def _x(rows, cols, seed=0, zero_rows=()):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((rows, cols)).astype(np.float32) * rng.uniform(0.01, 30, (rows, 1)).astype(np.float32)
    for r in zero_rows:
        v[r] = 0
    return gen.bf16_bits_from_f32(v)


def test_quant_act_mxfp8_bit_exact():
    x = _x(77, 4096, zero_rows=(3,))
    x[5, 64:96] = 0x8000  # a block of negative zeros
    xq, xs = gp.empty((77, 4096), torch.uint8), gp.empty((77, 128), torch.uint8)
    qb.qmoe_quant_act_mxfp8(gp.dev(x), xq, xs)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_act("mxfp4", x)
    assert np.array_equal(gp.host(xs), rs)
    assert np.array_equal(gp.host(xq), rq)


@pytest.mark.parametrize("src", ["bf16", "f32"])
def test_quant_rows_int8_bit_exact(src):
    rows, cols = 65, 1408
    xb = _x(rows, cols, seed=1, zero_rows=(7,))
    q, s = gp.empty((rows, cols), torch.int8), gp.empty(rows, torch.float32)
    if src == "bf16":
        qb.qmoe_quant_rows_int8_bf16(gp.dev(xb), q, s)
        xf = gp.bf16_to_f64(xb).astype(np.float32)
    else:
        xf = (np.random.default_rng(2).standard_normal((rows, cols)) * 3).astype(np.float32)
        xf[7] = 0
        qb.qmoe_quant_rows_int8_f32(gp.dev(xf), q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.int8_quant(xf)
    assert np.array_equal(gp.host(s), rs)
    assert np.array_equal(gp.host(q), rq)


# ------------------------------------------------------------------ stage 1

S1_CASES = [
    gen.custom("s1_w4a16", "w4a16", 40, 512, 6, 3, 256, seed=21),
    gen.custom("s1_w4a16_multitile", "w4a16", 200, 256, 3, 2, 128, seed=26),
    gen.custom("s1_mxfp4", "mxfp4", 40, 512, 6, 3, 384, seed=22),
    gen.custom("s1_mxfp4_tc", "mxfp4", 60, 512, 6, 3, 256, seed=24),
    gen.custom("s1_mxfp4_tc_multitile", "mxfp4", 200, 256, 3, 2, 128, seed=25),
    gen.custom("s1_w8a8", "w8a8", 40, 512, 6, 3, 256, seed=23),
    # K = 2304: two 1024-element drains and a 256-element tail
    gen.custom("s1_w8a8_drains", "w8a8", 120, 2304, 4, 2, 128, seed=27),
    # T*k > 96*E: 224-token schedule tiles, each run as two 112-token halves
    gen.custom("s1_w8a8_big_tiles", "w8a8", 500, 1280, 4, 2, 256, seed=28),
    gen.custom("s1_w4a8", "w4a8", 40, 512, 6, 3, 256, seed=29),
    # K = 2304 (18 steps), 224-token schedule tiles
    gen.custom("s1_w4a8_big_tiles", "w4a8", 500, 2304, 4, 2, 256, seed=30),
]


@pytest.mark.parametrize("w", S1_CASES, ids=[w.name for w in S1_CASES])
def test_stage1_against_oracle(w):
    d = gen.make_all(w)
    g = gp.run_layer(w, d, keep=True)
    ref_out, dbg, _ = oracle.moe_forward(w.scheme, dims(w), d, debug=True)
    ro = oracle.align_sort(d["topk_ids"], w.E)
    assert np.array_equal(g["sorted_pair_ids"], ro["sorted_pair_ids"])
    order = ro["sorted_pair_ids"]  # slot -> pair: oracle rows are pair-ordered
    if w.scheme == "w4a16":
        tok = order // w.k  # slot -> token
        # the permutation moves each bf16 row exactly: fp16 value * 2^e == the bf16 value
        xs = gp.bf16_to_f64(d["x"][tok])
        back = g["x_f16"].view(np.float16).astype(np.float64) * g["x_fac"][:, None].astype(np.float64)
        assert np.array_equal(back, xs)
        amax = np.abs(xs).max(axis=1)
        nz = amax > 0
        assert np.all((amax[nz] / g["x_fac"][nz] >= 2.0**14) & (amax[nz] / g["x_fac"][nz] < 2.0**15))
        got = gp.bf16_to_f64(g["h"])
        ref = gp.bf16_to_f64(dbg["hq"][order])
        assert rel_l2(got, ref) < W4_H_REL_L2
        # the tail holds each 32-column group's largest |h|
        assert np.array_equal(g["h_gmax"].astype(np.float64), np.abs(got).reshape(len(got), -1, 32).max(axis=2))
        # the down projection's fp16 form of h: the same values, each row scaled by its power of two
        back = g["h_f16"].view(np.float16).astype(np.float64) * g["h_fac"][:, None].astype(np.float64)
        assert np.array_equal(back, got)
        hmax = np.abs(got).max(axis=1)
        nz = hmax > 0
        assert np.all((hmax[nz] / g["h_fac"][nz] >= 2.0**14) & (hmax[nz] / g["h_fac"][nz] < 2.0**15))
    elif w.scheme == "mxfp4":
        rq, rs = oracle.quant_act("mxfp4", d["x"])
        tok = order // w.k  # slot -> token
        assert np.array_equal(g["xq"], rq[tok]) and np.array_equal(g["xs"], rs[tok])
        deq = lambda q, s: np.vectorize(oracle.e4m3_to_double)(q) * np.repeat(np.exp2(s.astype(np.float64) - 127),
                                                                              32, axis=1)
        got = deq(g["hq"], g["hs"])
        ref = deq(dbg["hq"][order], dbg["hs"][order])
        assert rel_l2(got, ref) < REL_L2
        assert np.mean(g["hq"] != dbg["hq"][order]) < 1e-3
    else:
        rq, rs = oracle.int8_quant(gp.bf16_to_f64(d["x"]).astype(np.float32))
        tok = order // w.k  # slot -> token
        assert np.array_equal(g["xq"], rq[tok]) and np.array_equal(g["xs"], rs[tok])
        assert np.array_equal(g["acc1"], dbg["acc1"][order])
        assert rel_l2(g["h"], dbg["h"][order]) < 1e-5
        # the intermediate codes follow the int8 rule on the kernel's own fp32 h
        hq, hs = oracle.int8_quant(g["h"].astype(np.float32))
        assert np.array_equal(g["hq"], hq) and np.array_equal(g["hs"], hs)
        # the tiles' per-(half tile, 128-step) maxima of sum |code|, which bound the GEMMs' fp32 partial sums
        nmax = gp.tile_nmax(w.T, w.k, w.E, w.H, w.I)
        nt = gp.max_tiles(w.P, w.E, nmax)
        t, r = gp._tile_index(g["offsets"], nmax, np.arange(g["offsets"][-1]))
        used = np.unique(t * (nmax // 112) + r // 112)
        for key, codes, K in (("x_l1", g["xq"], w.H), ("h_l1", g["hq"], w.I)):
            ref = gp.i8_step_l1max(codes, t, r, nmax, K, nt).reshape(-1, K // 128)
            assert np.array_equal(g[key].reshape(-1, K // 128)[used], ref[used]), key
    assert rel_l2(gp.bf16_to_f64(g["out"]), ref_out) < REL_L2


# ------------------------------------------------------------------ stage 2 on generator intermediates

S2_CASES = [
    gen.custom("s2_w4a16", "w4a16", 1, 512, 5, 1, 256, seed=31),
    gen.custom("s2_mxfp4", "mxfp4", 1, 768, 5, 1, 384, seed=32),
    gen.custom("s2_mxfp4_tc", "mxfp4", 1, 512, 5, 1, 256, seed=34),
    gen.custom("s2_w8a8", "w8a8", 1, 512, 5, 1, 256, seed=33),
    gen.custom("s2_w8a8_drains", "w8a8", 1, 256, 5, 1, 1152, seed=35),
    gen.custom("s2_w4a8", "w4a8", 1, 512, 5, 1, 1152, seed=36),
]


@pytest.mark.parametrize("w", S2_CASES, ids=[w.name for w in S2_CASES])
def test_stage2_against_oracle(w):
    rows = 300
    wts = gen.make_weights(w)
    s2 = gen.make_stage2_inputs(w, rows)
    experts = s2["experts"]
    counts = np.bincount(experts, minlength=w.E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    d = qb.dims(rows, 1, w.H, w.I, w.E)
    y = gp.empty((rows, w.H), torch.int16)  # bf16 bits
    t_off = gp.dev(offsets)
    yv = lambda: gp.bf16_to_f64(gp.host(y, np.uint16))
    if w.scheme == "w4a16":
        ids = experts.reshape(rows, 1)
        counts_t, off_t = gp.empty(w.E, torch.int32), gp.empty(w.E + 1, torch.int32)
        srt, slt = gp.empty(rows, torch.int32), gp.empty(rows, torch.int32)
        st = torch.zeros(1, dtype=torch.int32, device=gp.DEV)
        ws = qb.alloc_workspace(qb.workspace_bytes(d))
        qb.qmoe_align_sort(d, gp.dev(ids), counts_t, off_t, srt, slt, st, ws)
        nmax = gp.tile_nmax(rows, 1, w.E, w.H, w.I)
        ht = gp.pack_w4_h_tiles(s2["h"], offsets, nmax, w.I, qb.w4a16_h_tiles_bytes(d), gp.max_tiles(rows, w.E, nmax))
        w2p = qb.prepack_int4_weights(gp.dev(wts["w2"]), gp.dev(wts["w2_s"]), w.I)
        h16 = gp.empty(qb.w4a16_h16_tiles_bytes(d), torch.uint8)
        qb.qmoe_w4a16_h_to_f16(d, gp.dev(ht), off_t, h16, ws)
        qb.qmoe_gemm2_w4a16(d, h16, w2p, off_t, y, st, ws)
        ref = oracle.stage2("w4a16", w.H, w.I, w.E, experts, s2["h"], None, wts["w2"], wts["w2_s"])
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # y is stored as bf16: that rounding alone is ~1.1e-3 rel L2; the single
        # fp16 rounding of each dequantised weight adds ~2e-4 in quadrature
        assert rel_l2(yv(), ref) < Y_BF16_REL_L2
    elif w.scheme == "mxfp4":
        # the routing sort fills the workspace's tile schedule for these expert loads
        ids = experts.reshape(rows, 1)
        counts_t, off_t = gp.empty(w.E, torch.int32), gp.empty(w.E + 1, torch.int32)
        srt, slt = gp.empty(rows, torch.int32), gp.empty(rows, torch.int32)
        st = torch.zeros(1, dtype=torch.int32, device=gp.DEV)
        ws = qb.alloc_workspace(qb.workspace_bytes(d))
        qb.qmoe_align_sort(d, gp.dev(ids), counts_t, off_t, srt, slt, st, ws)
        ht = gp.pack_tiles(s2["h"], s2["h_s"], offsets, gp.tile_nmax(rows, 1, w.E, w.H, w.I), w.I, qb.mx_tiles_bytes(d, w.I))
        w2p = qb.prepack_mx_scales(gp.dev(wts["w2_s"]), w.I)
        w2w = qb.prepack_fp4_weights(gp.dev(wts["w2"]), w.I)
        qb.qmoe_gemm2_mxfp4(d, gp.dev(ht), w2w, w2p, off_t, y, st, ws)
        ref = oracle.stage2("mxfp4", w.H, w.I, w.E, experts, s2["h"], s2["h_s"], wts["w2"], wts["w2_s"])
        torch.cuda.synchronize()
        # every E2M1 x E4M3 product and its scales are exact in fp32; the only
        # roundings are the tensor core's sum and y's bf16 rounding.  Per
        # element: within one bf16 step of the double sum, plus a sum error of
        # at most 2^-16 of the terms' absolute sum (a sum that cancels can sit
        # far below its terms)
        got = yv()
        hv = torch.from_numpy(s2["h"]).view(torch.float8_e4m3fn).double().numpy() * \
            np.repeat(np.exp2(s2["h_s"].astype(np.float64) - 127.0), 32, axis=1)
        W2 = bf.dequant_w("mxfp4", wts["w2"], wts["w2_s"])
        A = np.einsum("rk,rnk->rn", np.abs(hv), np.abs(W2[experts]))
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
        excess = (np.abs(got - ref) - ulp) / np.maximum(A, 1e-300)
        assert excess.max() <= 2.0 ** -16, f"excess over one bf16 step: {excess.max():.3e} of the terms' |sum|"
        assert rel_l2(got, ref) < Y_BF16_REL_L2
    else:
        ids = experts.reshape(rows, 1)
        counts_t, off_t = gp.empty(w.E, torch.int32), gp.empty(w.E + 1, torch.int32)
        srt, slt = gp.empty(rows, torch.int32), gp.empty(rows, torch.int32)
        st = torch.zeros(1, dtype=torch.int32, device=gp.DEV)
        ws = qb.alloc_workspace(qb.workspace_bytes(d))
        qb.qmoe_align_sort(d, gp.dev(ids), counts_t, off_t, srt, slt, st, ws)
        nmax = gp.tile_nmax(rows, 1, w.E, w.H, w.I)
        ht = gp.pack_i8_tiles(s2["h"], s2["h_s"], offsets, nmax, w.I, qb.w8a8_tiles_bytes(d, w.I),
                              gp.max_tiles(rows, w.E, nmax))
        acc = gp.empty((rows, w.H), torch.int32)
        g2 = qb.qmoe_gemm2_w8a8 if w.scheme == "w8a8" else qb.qmoe_gemm2_w4a8
        g2(d, gp.dev(ht), gp.dev(wts["w2"]), gp.dev(wts["w2_s"]), off_t, y, acc, st, ws)
        ref, racc = oracle.stage2(w.scheme, w.H, w.I, w.E, experts, s2["h"], s2["h_s"], wts["w2"], wts["w2_s"],
                                  acc=True)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(gp.host(acc), racc)
        # y = ((float)acc * s_h) * s_w is exact fp32 on both sides; both round it to bf16
        ref_bf16 = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(gp.host(y), ref_bf16)


def _stage2_int_direct(w, h, hs, w2, w2s, experts):
    """Stage 2 alone on given int8 codes (slot order, experts ascending)."""
    rows = len(h)
    counts = np.bincount(experts, minlength=w.E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    d = qb.dims(rows, 1, w.H, w.I, w.E)
    counts_t, off_t = gp.empty(w.E, torch.int32), gp.empty(w.E + 1, torch.int32)
    srt, slt = gp.empty(rows, torch.int32), gp.empty(rows, torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device=gp.DEV)
    ws = qb.alloc_workspace(qb.workspace_bytes(d))
    qb.qmoe_align_sort(d, gp.dev(experts.reshape(rows, 1).astype(np.int32)), counts_t, off_t, srt, slt, st, ws)
    nmax = gp.tile_nmax(rows, 1, w.E, w.H, w.I)
    ht = gp.pack_i8_tiles(h, hs, offsets, nmax, w.I, qb.w8a8_tiles_bytes(d, w.I), gp.max_tiles(rows, w.E, nmax))
    y, acc = gp.empty((rows, w.H), torch.int16), gp.empty((rows, w.H), torch.int32)
    g2 = qb.qmoe_gemm2_w8a8 if w.scheme == "w8a8" else qb.qmoe_gemm2_w4a8
    g2(d, gp.dev(ht), gp.dev(w2), gp.dev(w2s), off_t, y, acc, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return gp.host(acc)


@pytest.mark.parametrize("K", [1024, 4096, 16384])
def test_w8a8_adversarial_accumulators_exact(K):
    # all-+-127 operands: the largest-magnitude int32 sums a row of length K makes
    # (127^2 * 4096 = 66,064,384 is far past 2^24, where fp32 stops being exact;
    # at K = 16384, the largest supported, the carried high parts reach 32,258 of
    # their 16-bit range)
    w = gen.custom("adv", "w8a8", 1, 256, 2, 1, K, seed=5)
    rows = 64
    h = np.full((rows, w.I), 127, np.int8)
    h[1::2] = -127
    w2 = np.full((w.E, w.H, w.I), 127, np.int8)
    w2[:, ::3] = -127
    hs = np.full(rows, 1e-3, np.float32)
    w2s = np.full((w.E, w.H), 1e-3, np.float32)
    experts = np.repeat(np.arange(w.E, dtype=np.int32), rows // w.E)
    got = _stage2_int_direct(w, h, hs, w2, w2s, experts)
    _, racc = oracle.stage2("w8a8", w.H, w.I, w.E, experts, h, hs, w2, w2s, acc=True)
    assert np.array_equal(got, racc)
    assert np.abs(racc).max() == 127 * 127 * w.I


def test_w4a8_extreme_codes_exact_at_largest_K():
    # every |h| = 127 against every |code| = 7 at K = 16384: partial sums up to
    # 7 * 127 * 16384, just under 2^24, with no carry passes
    K = 16384
    w = gen.custom("adv4", "w4a8", 1, 256, 2, 1, K, seed=8)
    rng = np.random.default_rng(8)
    rows = 40
    experts = np.sort(rng.integers(0, w.E, size=rows)).astype(np.int32)
    h = np.where(rng.random((rows, K)) < 0.5, 127, -127).astype(np.int8)
    h[: rows // 2] = 127  # half the rows all +127: sums of one sign
    hs = np.full(rows, 1e-3, np.float32)
    # nibbles 1 (code -7) or 15 (code +7); the first expert's first rows all +7
    nib = np.where(rng.random((w.E, w.H, K)) < 0.5, 1, 15).astype(np.uint8)
    nib[0, :16] = 15
    w2 = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    w2s = np.full((w.E, w.H), 1e-3, np.float32)
    got = _stage2_int_direct(w, h, hs, w2, w2s, experts)
    _, racc = oracle.stage2("w4a8", w.H, w.I, w.E, experts, h, hs, w2, w2s, acc=True)
    assert np.array_equal(got, racc)
    assert np.abs(racc).max() >= 7 * 127 * K - 14 * 127 * 64


def test_w8a8_stage1_adversarial_accumulators_exact():
    # every activation code +-127 and every weight +-127 along K = H = 4096
    w = gen.custom("adv1", "w8a8", 8, 4096, 2, 1, 128, seed=6)
    d = gen.make_all(w)
    sign = np.where(np.arange(w.H) % 5 == 0, -1.0, 1.0).astype(np.float32)
    d["x"] = gen.bf16_bits_from_f32(np.tile(sign, (w.T, 1)) * np.arange(1, w.T + 1, dtype=np.float32)[:, None])
    w1 = np.where(np.arange(w.H) % 5 == 0, -127, 127).astype(np.int8)
    d["w1"] = np.tile(w1, (w.E, 2 * w.I, 1))
    d["w1"][:, 1::2] *= -1
    d["w1_s"] = np.full((w.E, 2 * w.I), 1e-9, np.float32)
    g = gp.run_layer(w, d, keep=True)
    _, dbg, _ = oracle.moe_forward(w.scheme, dims(w), d, debug=True)
    order = oracle.align_sort(d["topk_ids"], w.E)["sorted_pair_ids"]
    assert np.array_equal(g["acc1"], dbg["acc1"][order])
    assert np.abs(dbg["acc1"]).max() == 127 * 127 * w.H


# ------------------------------------------------------------------ combine

def test_combine_against_oracle_and_deterministic():
    T, k, H = 300, 10, 1024
    rng = np.random.default_rng(9)
    ids = gen.routing_uniform(rng, T, 64, k)
    ids[5, 3] = 99  # one invalid pair: slot -1
    ro = oracle.align_sort(ids, 64)
    y = gen.bf16_bits_from_f32(rng.standard_normal((T * k, H)).astype(np.float32))
    tw = gen.routing_weights(rng, T, k)
    d = qb.dims(T, k, H, 32, 64)
    outs = []
    for _ in range(2):
        out = gp.empty((T, H), torch.int16)
        qb.qmoe_combine(d, gp.dev(y), gp.dev(tw), gp.dev(ro["pair_slot"]), out)
        torch.cuda.synchronize()
        outs.append(gp.host(out, np.uint16))
    assert np.array_equal(outs[0], outs[1])
    ref = oracle.combine(gp.bf16_to_f64(y).astype(np.float32), tw, ro["pair_slot"])
    assert rel_l2(gp.bf16_to_f64(outs[0]), ref) < REL_L2


# ------------------------------------------------------------------ whole layer

SMALL = [
    gen.WORKLOADS["tiny_w4a16"],
    gen.custom("e2e_mxfp4_ragged", "mxfp4", 50, 1024, 12, 4, 128, seed=41),
    gen.custom("e2e_w8a8_ragged", "w8a8", 50, 1024, 12, 4, 256, seed=42),
    gen.custom("e2e_w4a8_ragged", "w4a8", 50, 1024, 12, 4, 256, seed=48),
    gen.custom("e2e_w4a16_ragged", "w4a16", 50, 1024, 12, 4, 256, seed=43),
    gen.custom("e2e_w4a16_big_tiles", "w4a16", 700, 512, 8, 2, 256, seed=47),
    gen.custom("e2e_zipf_mxfp4", "mxfp4", 64, 512, 64, 8, 128, routing="zipf", seed=44),
    gen.custom("e2e_mxfp4_tc", "mxfp4", 96, 1024, 16, 4, 384, seed=45),
    gen.custom("e2e_mxfp4_tc_big_tiles", "mxfp4", 700, 512, 8, 2, 256, seed=46),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_layer_small(w):
    d = gen.make_all(w)
    g = gp.run_layer(w, d)
    ref = oracle.moe_forward(w.scheme, dims(w), d)
    assert g["status"] == 0
    assert rel_l2(gp.bf16_to_f64(g["out"]), ref) < REL_L2


@pytest.mark.parametrize("scheme", ["mxfp4", "w8a8"])
@pytest.mark.parametrize("k", [33, 40])
def test_layer_topk_above_32(scheme, k):
    # the token-major permutes walk a token's pairs 32 at a time and the combine
    # 8 at a time: k = 33 and 40 run both loops past their first chunk, with a
    # ragged last chunk ([hip-ep] description: fixed-order scatter back)
    w = gen.custom(f"topk{k}_{scheme}", scheme, 24, 512, 48, k, 128, seed=90 + k)
    d = gen.make_all(w)
    g = gp.run_layer(w, d)
    ref = oracle.moe_forward(w.scheme, dims(w), d)
    assert g["status"] == 0
    assert rel_l2(gp.bf16_to_f64(g["out"]), ref) < REL_L2
    wt = gp.device_weights(w, d)
    out, status = qb.moe_forward(scheme, gp.dev(d["x"]), gp.dev(d["topk_ids"]), gp.dev(d["topk_w"]),
                                 wt["w1"], wt["w1_s"], wt["w2"], wt["w2_s"], I=w.I, E=w.E)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(gp.host(out, np.uint16), g["out"])


@pytest.mark.parametrize("scheme", ["w4a16", "mxfp4", "w8a8", "w4a8"])
def test_layer_ragged_expert_loads(scheme):
    # expert loads 0, 1, 127, 129 (tile tails on both sides of 128) plus empties
    counts = [0, 1, 127, 129, 0, 3, 0, 4]
    rng = np.random.default_rng(77)
    ids = gen.routing_with_counts(rng, counts, 2)
    T = ids.shape[0]
    w = gen.custom(f"ragged_{scheme}", scheme, T, 256, len(counts), 2, 128, seed=78)  # H % 256, I % 128
    d = gen.make_all(w, routing=(ids, gen.routing_weights(rng, T, 2)))
    g = gp.run_layer(w, d)
    ref = oracle.moe_forward(scheme, dims(w), d)
    assert rel_l2(gp.bf16_to_f64(g["out"]), ref) < REL_L2


def test_layer_invalid_ids_flagged_and_skipped():
    w = gen.custom("bad_ids", "mxfp4", 20, 256, 8, 2, 128, seed=51)
    d = gen.make_all(w)
    d["topk_ids"] = d["topk_ids"].copy()
    d["topk_ids"][3, 1] = 8
    d["topk_ids"][7, 0] = -2
    g = gp.run_layer(w, d)
    ref = oracle.moe_forward(w.scheme, dims(w), d)
    assert g["status"] & qb.DEV_BAD_EXPERT_ID
    assert rel_l2(gp.bf16_to_f64(g["out"]), ref) < REL_L2


@pytest.mark.parametrize("nmax", [16, 112, 224])
def test_mxfp4_stage1_gather_equals_permuted_tiles(nmax):
    # Stage 1 reading token-major MX x through the routing order writes the same h tiles, bit for
    # bit, as stage 1 reading the permuted tiles: expert loads on both sides of each tile size,
    # empty experts, and two invalid expert ids (pairs without a slot)
    counts = [0, 1, 15, 16, 17, 0, 111, 112, 113, 223, 225, 3]
    rng = np.random.default_rng(95)
    ids = gen.routing_with_counts(rng, counts, 2)
    ids[1, 0], ids[5, 1] = len(counts), -1
    T, k, H, I, E = ids.shape[0], 2, 512, 256, len(counts)
    w = gen.custom(f"gather{nmax}", "mxfp4", T, H, E, k, I, seed=96)
    d = gen.make_all(w, routing=(ids, gen.routing_weights(rng, T, k)))
    dd = qb.dims(T, k, H, I, E)
    t = {key: gp.dev(v) for key, v in d.items()}
    try:
        qb.set_tile_rules([dict(H=H, I=I, E=E, k=k, t_min=T, t_max=T, nmax=nmax)])
        assert qb.tile_nmax(dd) == nmax
        P = T * k
        counts_d, offsets = gp.empty(E, torch.int32), gp.empty(E + 1, torch.int32)
        sorted_ids, slot = gp.empty(P, torch.int32), gp.empty(P, torch.int32)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = qb.alloc_workspace(qb.workspace_bytes(dd))
        qb.qmoe_align_sort(dd, t["topk_ids"], counts_d, offsets, sorted_ids, slot, status, ws)
        w1, w1p, _, _ = qb.prepack_mxfp4(t["w1"], t["w1_s"], t["w2"], t["w2_s"], H, I)
        xt = gp.empty(qb.mx_tiles_bytes(dd, H), torch.uint8)
        qb.qmoe_permute_quant_mxfp8(dd, t["x"], slot, offsets, xt, ws)
        h_tiles = torch.zeros(qb.mx_tiles_bytes(dd, I), dtype=torch.uint8, device="cuda")
        qb.qmoe_gemm1_swiglu_mxfp4(dd, xt, w1, w1p, offsets, h_tiles, status, ws)
        xq, xs = gp.empty((T, H), torch.uint8), gp.empty((T, H // 32), torch.uint8)
        qb.qmoe_quant_act_mxfp8(t["x"], xq, xs)
        h_gather = torch.zeros_like(h_tiles)
        qb.qmoe_gemm1_swiglu_mxfp4_gather(dd, xq, xs, sorted_ids, w1, w1p, offsets, h_gather, status, ws)
        torch.cuda.synchronize()
    finally:
        qb.set_tile_rules(qb.read_tile_table(qb.TILE_TABLE_PATH) if os.path.exists(qb.TILE_TABLE_PATH) else [])
    assert int(status.item()) == qb.DEV_BAD_EXPERT_ID  # the sort flags the two ids; nothing else
    assert np.array_equal(gp.host(h_gather), gp.host(h_tiles))
    assert gp.host(h_gather).any()


def test_layer_zero_tokens():
    w = gen.custom("empty", "w4a16", 0, 256, 8, 2, 128, seed=1)
    d = gen.make_all(w)
    wt = gp.device_weights(w, d)
    out, status = qb.moe_forward("w4a16", gp.empty((0, 256), torch.int16), gp.empty((0, 2), torch.int32),
                                 gp.empty((0, 2), torch.float32), wt["w1"], None, wt["w2"], None, I=w.I, E=w.E)
    torch.cuda.synchronize()
    assert out.shape == (0, 256) and int(status.item()) == 0


@pytest.mark.parametrize("scheme", ["w4a16", "mxfp4", "w8a8", "w4a8"])
def test_forward_entry_point_matches_stagewise_and_is_deterministic(scheme):
    w = gen.custom(f"fwd_{scheme}", scheme, 33, 512, 10, 4, 128, seed=61)  # I, H multiples of 128
    d = gen.make_all(w)
    stage = gp.run_layer(w, d)
    outs = []
    wt = gp.device_weights(w, d)
    for _ in range(2):
        out, status = qb.moe_forward(scheme, gp.dev(d["x"]), gp.dev(d["topk_ids"]), gp.dev(d["topk_w"]),
                                     wt["w1"], wt["w1_s"], wt["w2"], wt["w2_s"], I=w.I, E=w.E)
        torch.cuda.synchronize()
        outs.append(gp.host(out, np.uint16))
        assert int(status.item()) == 0
    assert np.array_equal(outs[0], outs[1])
    assert np.array_equal(outs[0], stage["out"])


@pytest.mark.parametrize("scheme", ["w4a16", "mxfp4", "w8a8", "w4a8"])
def test_forward_back_to_back_calls_share_a_workspace(scheme):
    # Consecutive whole-layer calls on one stream, no synchronisation between
    # them, one workspace: each kernel may start before the one ahead of it
    # completes (dependent launches), and the next call's routing sort
    # rewrites the buffers the previous call's combine reads.  Every call must
    # still equal the same batch run alone, stage by stage.
    H, E, k, I = 512, 10, 4, 256
    ws_ = [gen.Workload(f"b2b_{scheme}_{i}", scheme, T, H, E, k, I, "uniform", 300 + i, 299)
           for i, T in enumerate((40, 7, 33, 1))]
    ds = [gen.make_all(w) for w in ws_]
    wt = gp.device_weights(ws_[0], ds[0])
    qd = lambda w: qb.dims(w.T, w.k, w.H, w.I, w.E)
    ws = qb.alloc_workspace(max(qb.forward_workspace_bytes(qd(w), scheme) for w in ws_))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ins = [{key: gp.dev(d[key]) for key in ("x", "topk_ids", "topk_w")} for d in ds]
    outs = [gp.empty((w.T, H), torch.int16) for w in ws_]
    torch.cuda.synchronize()
    for _ in range(2):
        for w, t, out in zip(ws_, ins, outs):
            qb.qmoe_moe_forward(scheme, qd(w), t["x"], t["topk_ids"], t["topk_w"], wt["w1"], wt["w1_s"], wt["w2"],
                                wt["w2_s"], out, status, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for w, d, out in zip(ws_, ds, outs):
        assert np.array_equal(gp.host(out, np.uint16), gp.run_layer(w, d)["out"]), w.name


def test_forward_switches_mxfp4_stage1_form_between_calls():
    # The whole-layer call gathers x in stage 1 for some shapes and reads permuted tiles for
    # others (qmoe_mx_layer_gathers).  Calls of both kinds back to back on one stream and one
    # workspace, no synchronisation between them: each equals its batch run through the stage
    # calls (permuted tiles), bit for bit.
    H, E, k, I = 512, 8, 4, 256
    ws_ = [gen.Workload(f"sw_{i}", "mxfp4", T, H, E, k, I, "uniform", 400 + i, 399)
           for i, T in enumerate((200, 7, 161, 40))]
    qd = lambda w: qb.dims(w.T, w.k, w.H, w.I, w.E)
    assert [qb.mx_layer_gathers(qd(w)) for w in ws_] == [True, False, True, False]
    ds = [gen.make_all(w) for w in ws_]
    wt = gp.device_weights(ws_[0], ds[0])
    ws = qb.alloc_workspace(max(qb.forward_workspace_bytes(qd(w), "mxfp4") for w in ws_))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ins = [{key: gp.dev(d[key]) for key in ("x", "topk_ids", "topk_w")} for d in ds]
    outs = [gp.empty((w.T, H), torch.int16) for w in ws_]
    torch.cuda.synchronize()
    for _ in range(2):
        for w, t, out in zip(ws_, ins, outs):
            qb.qmoe_moe_forward("mxfp4", qd(w), t["x"], t["topk_ids"], t["topk_w"], wt["w1"], wt["w1_s"], wt["w2"],
                                wt["w2_s"], out, status, ws)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for w, d, out in zip(ws_, ds, outs):
        assert np.array_equal(gp.host(out, np.uint16), gp.run_layer(w, d)["out"]), w.name


def test_forward_16row_tiles_back_to_back_with_unrouted_token():
    # The whole-layer MXFP4 call with 16-row token tiles (the decode form) against the stage calls,
    # bit for bit: ragged loads, invalid ids (one token with none of its pairs routed, whose row must
    # come out zero), calls of several sizes back to back on one workspace, outputs pre-filled with
    # NaN so no row is left unwritten.
    H, E, k, I = 512, 12, 4, 256
    ws_ = [gen.Workload(f"fz_{i}", "mxfp4", T, H, E, k, I, "uniform", 500 + i, 499)
           for i, T in enumerate((37, 5, 1, 16))]
    ds = [gen.make_all(w) for w in ws_]
    ds[0]["topk_ids"] = ds[0]["topk_ids"].copy()
    ds[0]["topk_ids"][3, :] = -1
    ds[0]["topk_ids"][7, 2] = E
    qd = lambda w: qb.dims(w.T, w.k, w.H, w.I, w.E)
    try:
        qb.set_tile_rules([dict(H=H, I=I, E=E, k=k, t_min=1, t_max=64, nmax=16)])
        for w in ws_:
            assert qb.tile_nmax(qd(w)) == 16 and qb.forward_launches(qd(w), "mxfp4") == 5
        wt = gp.device_weights(ws_[0], ds[0])
        ws = qb.alloc_workspace(max(qb.forward_workspace_bytes(qd(w), "mxfp4") for w in ws_))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ins = [{key: gp.dev(d[key]) for key in ("x", "topk_ids", "topk_w")} for d in ds]
        outs = [torch.full((w.T, H), 0x7FC0, dtype=torch.int16, device="cuda") for w in ws_]
        torch.cuda.synchronize()
        for _ in range(2):
            for w, t, out in zip(ws_, ins, outs):
                qb.qmoe_moe_forward("mxfp4", qd(w), t["x"], t["topk_ids"], t["topk_w"], wt["w1"], wt["w1_s"],
                                    wt["w2"], wt["w2_s"], out, status, ws)
        torch.cuda.synchronize()
        refs = [gp.run_layer(w, d) for w, d in zip(ws_, ds)]
    finally:
        qb.set_tile_rules(qb.read_tile_table(qb.TILE_TABLE_PATH) if os.path.exists(qb.TILE_TABLE_PATH) else [])
    assert int(status.item()) == qb.DEV_BAD_EXPERT_ID
    for w, out, ref in zip(ws_, outs, refs):
        assert np.array_equal(gp.host(out, np.uint16), ref["out"]), w.name
    assert not refs[0]["out"][3].any()  # the token with no routed pair


@pytest.mark.parametrize("scheme", ["mxfp4", "w8a8", "w4a8", "w4a16"])
@pytest.mark.parametrize("nmax", [16, 112, 224])
def test_layer_with_each_token_tile(scheme, nmax):
    # the tile table may pick either token tile for any shape: both match the oracle
    w = gen.custom(f"tile{nmax}_{scheme}", scheme, 150, 512, 6, 4, 256, seed=81)  # ~100 pairs per expert
    d = gen.make_all(w)
    try:
        qb.set_tile_rules([dict(H=w.H, I=w.I, E=w.E, k=w.k, t_min=w.T, t_max=w.T, nmax=nmax)])
        assert qb.tile_nmax(qb.dims(w.T, w.k, w.H, w.I, w.E)) == nmax
        g = gp.run_layer(w, d, keep=True)
    finally:
        qb.set_tile_rules(qb.read_tile_table(qb.TILE_TABLE_PATH) if os.path.exists(qb.TILE_TABLE_PATH) else [])
    ref = oracle.moe_forward(w.scheme, dims(w), d)
    assert g["status"] == 0
    assert rel_l2(gp.bf16_to_f64(g["out"]), ref) < REL_L2


@pytest.mark.parametrize("scheme", ["w4a16", "w8a8", "w4a8", "mxfp4"])
def test_layer_token_halves_at_their_edges(scheme):
    # 224-row tiles: the integer GEMMs split a tile into token halves (112 + 112, or 160 + 64 for
    # W4A16) and enumerate only the non-empty ones; expert loads just below, at and above each
    # half and tile boundary, plus empty experts between them
    counts = [0, 1, 111, 112, 113, 0, 159, 160, 161, 224, 225, 0, 335, 336, 449]
    rng = np.random.default_rng(91)
    ids = gen.routing_with_counts(rng, counts, 1)
    T = ids.shape[0]
    w = gen.custom(f"halves_{scheme}", scheme, T, 256, len(counts), 1, 128, seed=92)  # H % 256, I % 128
    d = gen.make_all(w, routing=(ids, gen.routing_weights(rng, T, 1)))
    try:
        qb.set_tile_rules([dict(H=w.H, I=w.I, E=w.E, k=w.k, t_min=w.T, t_max=w.T, nmax=224)])
        assert qb.tile_nmax(qb.dims(w.T, w.k, w.H, w.I, w.E)) == 224
        g = gp.run_layer(w, d, keep=True)
    finally:
        qb.set_tile_rules(qb.read_tile_table(qb.TILE_TABLE_PATH) if os.path.exists(qb.TILE_TABLE_PATH) else [])
    ref = oracle.moe_forward(w.scheme, dims(w), d)
    assert g["status"] == 0
    assert rel_l2(gp.bf16_to_f64(g["out"]), ref) < REL_L2
    # every routed token's output row is produced (no unit skipped)
    assert (np.abs(gp.bf16_to_f64(g["out"])).max(axis=1) > 0).all()


def test_argument_errors_raise():
    w = gen.custom("err", "w4a16", 4, 256, 4, 2, 64, seed=1)
    d = gen.make_all(w)
    with pytest.raises(qb.QmoeError):
        qb.qmoe_combine(qb.dims(4, 2, 250, 64, 4), gp.empty((8, 250), torch.float32), gp.dev(d["topk_w"]),
                        gp.empty(8, torch.int32), gp.empty((4, 250), torch.int16))


# ------------------------------------------------------------------ full-size workloads (sampled rows)

_WEIGHT_CACHE = {}


def _full_inputs(w):
    key = (w.scheme, w.H, w.I, w.E, w.wseed)
    if key not in _WEIGHT_CACHE:
        _WEIGHT_CACHE.clear()
        _WEIGHT_CACHE[key] = gen.make_weights(w)
    ids, tw = gen.make_routing(w)
    d = dict(x=gen.make_activations(w), topk_ids=ids, topk_w=tw)
    d.update(_WEIGHT_CACHE[key])
    return d


FULL = ["decode_T1", "decode_T4", "decode_T16", "decode_T64", "mxfp4_T256", "mxfp4_T1024", "mxfp4_T4096",
        "mxfp4_T8192", "w4a16_T2048", "w8a8_T8192", "w4a8_T8192",
        # tensor-parallel shards: inter 512 (TP2) and 256 (TP4)
        "mxfp4_tp2_T4096", "mxfp4_tp2_T8192", "mxfp4_tp4_T16", "mxfp4_tp4_T4096"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name):
    w = gen.WORKLOADS[name]
    d = _full_inputs(w)
    g = gp.run_layer(w, d)
    assert g["status"] == 0
    n = min(w.T, 48)
    rows = np.sort(np.random.default_rng(w.seed).choice(w.T, n, replace=False))
    ref = oracle.moe_forward(w.scheme, dims(w), d, tokens=rows)
    assert rel_l2(gp.bf16_to_f64(g["out"][rows]), ref) < REL_L2
    # every row is finite and the layer is not trivially zero
    allout = gp.bf16_to_f64(g["out"])
    assert np.isfinite(allout).all() and np.abs(allout).max() > 0
    # the whole-layer call, launched as bench.py times it (dependent launches, weights read before the
    # wait on the previous kernel, L2 prefetches), gives the same bits as the stage calls
    wt = gp.device_weights(w, d)
    out, status = qb.moe_forward(w.scheme, gp.dev(d["x"]), gp.dev(d["topk_ids"]), gp.dev(d["topk_w"]), wt["w1"],
                                 wt["w1_s"], wt["w2"], wt["w2_s"], I=w.I, E=w.E)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(gp.host(out, np.uint16), g["out"])


def test_w4a16_unsupported_shapes_rejected_on_host():
    # the W4A16 tensor-core path needs H % 256 == 0 and I % 128 == 0
    d = qb.dims(8, 2, 256, 96, 4)
    x = gp.empty(qb.w4a16_x_tiles_bytes(d), torch.uint8)
    ws = qb.alloc_workspace(qb.workspace_bytes(d))
    st = torch.zeros(1, dtype=torch.int32, device=gp.DEV)
    w = gp.empty(1 << 16, torch.uint8)
    with pytest.raises(qb.QmoeError, match="-2"):
        qb.qmoe_gemm1_swiglu_w4a16(d, x, w, gp.empty(5, torch.int32), x, st, ws)


def test_int4_prepack_layout():
    # pre-packed blocks against the layout stated in include/qmoe.h, built here in numpy
    rng = np.random.default_rng(5)
    rows, K = 200, 160
    w = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    s = rng.integers(0, 0x7C00, (rows, K // 32), dtype=np.uint16)
    s[7] = 0  # an all-zero row keeps factor 1
    s[9] = 0x0001  # the smallest fp16 subnormal: the row's factor is 2^-34
    got = gp.host(qb.prepack_int4_weights(gp.dev(w), gp.dev(s), K))
    KT, RT = (K + 63) // 64, (rows + 127) // 128
    assert got.size == RT * KT * 4608 + RT * 128 * 4
    nib = np.zeros((RT * 128, KT * 64), np.uint8) + 8
    nib[:rows, :K] = np.stack([w & 15, w >> 4], axis=-1).reshape(rows, K)
    sv = s.view(np.float16).astype(np.float64)
    smax = np.abs(sv).max(axis=1)
    p = np.where(smax > 0, 10 - np.floor(np.log2(np.where(smax > 0, smax, 1))), 0)
    fac = got[RT * KT * 4608:].view(np.float32)
    assert np.array_equal(fac[:rows].astype(np.float64), np.exp2(-p)) and np.all(fac[rows:] == 1)
    assert fac[9] == 2.0**-34 and fac[7] == 1
    scaled = np.zeros((RT * 128, KT * 2), np.float64)
    # fp16 values times powers of two, rounded back to fp16 (only scales far below their row's largest, which
    # become fp16 subnormals, round)
    scaled[:rows, :K // 32] = (sv * np.exp2(p)[:, None]).astype(np.float16).astype(np.float64)
    words = got[:RT * KT * 4608].view(np.uint32)
    for rt in range(RT):
        for kt in range(KT):
            blk = words[(rt * KT + kt) * 1152:(rt * KT + kt + 1) * 1152]
            codes = blk[:1024].reshape(128, 8)
            for m in range(8):  # element m of each 8-element word
                pos = 4 + m // 2 if m % 2 else m // 2
                ref = nib[rt * 128:(rt + 1) * 128, kt * 64 + m:kt * 64 + 64:8]
                assert np.array_equal((codes >> np.uint32(4 * pos)) & 15, ref)
            sw = blk[1024:]
            lo = (sw & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
            hi = (sw >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
            assert np.array_equal(lo, scaled[rt * 128:(rt + 1) * 128, 2 * kt])
            assert np.array_equal(hi, scaled[rt * 128:(rt + 1) * 128, 2 * kt + 1])
    assert np.abs(scaled).max() < 2.0**11


def test_mxfp4_unsupported_shapes_rejected_on_host():
    # the MXFP4 tensor-core path needs H % 256 == 0 and I % 128 == 0
    d = qb.dims(8, 2, 384, 128, 4)
    x = gp.empty(qb.mx_tiles_bytes(d, 384) or 16, torch.uint8)
    ws = qb.alloc_workspace(qb.workspace_bytes(d))
    st = torch.zeros(1, dtype=torch.int32, device=gp.DEV)
    w = gp.empty(1 << 16, torch.uint8)
    with pytest.raises(qb.QmoeError, match="-2"):
        qb.qmoe_gemm1_swiglu_mxfp4(d, x, w, w, gp.empty(5, torch.int32), x, st, ws)
