"""CPU checks of the C ABI: the CUDA library loads, exports every function
include/qmoe.h declares, and rejects bad arguments on the host before any
launch (these calls touch no GPU)."""

import ctypes
import glob
import os
import re

import pytest

from quantized_mixture_experts_moe_gb300 import binding as qb
from quantized_mixture_experts_moe_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(qmoe_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qb.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["qmoe_align_sort", "qmoe_gemm1_swiglu_w4a16", "qmoe_gemm1_swiglu_mxfp4", "qmoe_gemm1_swiglu_w8a8",
                     "qmoe_gemm2_w4a16", "qmoe_gemm2_mxfp4", "qmoe_gemm2_w8a8", "qmoe_combine"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) <= set(qb.SIGNATURES)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4):
        assert qb.status_str(code)
    assert "sm_103a" in qb.version()


def test_workspace_bytes_host_only(lib):
    d = qb.dims(4096, 10, 4096, 1024, 512)
    n = qb.workspace_bytes(d)
    assert n >= 4 * 512 * ((40960 + 2047) // 2048)
    # plus the tile schedule (E + 1 ints) and one token-tile row per slot and per pair
    assert n >= 4 * 512 * ((40960 + 2047) // 2048) + 4 * 513 + 2 * 4 * 40960
    # holds y (bf16, slot order) and the token-major MX x (codes and scales)
    assert qb.forward_workspace_bytes(d, "mxfp4") > 40960 * 4096 * 2 + 4096 * 4096 * 33 // 32
    bad = qb.dims(16, 2, 250, 128, 8)  # H not a multiple of 32
    assert qb.workspace_bytes(bad) == 0


def test_mx_layer_stage1_choice_host_only(lib):
    # the whole-layer call gathers x in MXFP4 stage 1 only with 112/224-row tiles, I <= 512 and
    # at least 64 pairs per expert; host-only, no GPU needed
    rules = qb.read_tile_table(qb.TILE_TABLE_PATH) if os.path.exists(qb.TILE_TABLE_PATH) else []
    try:
        qb.set_tile_rules([])  # built-in tile rule: 224 rows above 96 pairs per expert, else 112
        assert qb.mx_layer_gathers(qb.dims(4096, 10, 4096, 256, 512))      # 80 pairs per expert, 112 rows
        assert qb.mx_layer_gathers(qb.dims(8192, 10, 4096, 512, 512))      # 160 per expert, 224 rows
        assert not qb.mx_layer_gathers(qb.dims(4096, 10, 4096, 1024, 512))  # I 1024
        assert not qb.mx_layer_gathers(qb.dims(1024, 10, 4096, 256, 512))   # 20 pairs per expert
        qb.set_tile_rules([dict(H=4096, I=256, E=512, k=10, t_min=1, t_max=8192, nmax=16)])
        assert not qb.mx_layer_gathers(qb.dims(4096, 10, 4096, 256, 512))  # 16-row tiles
        assert not qb.mx_layer_gathers(qb.dims(16, 2, 250, 128, 8))         # invalid dims
    finally:
        qb.set_tile_rules(rules)


def test_forward_launch_count_host_only(lib):
    # kernels one whole-layer call launches: routing sort (1 up to 2048 pairs, else 2), activation
    # quantisation, two GEMMs, the W4A16 / integer intermediate pass, and the combine
    rules = qb.read_tile_table(qb.TILE_TABLE_PATH) if os.path.exists(qb.TILE_TABLE_PATH) else []
    try:
        qb.set_tile_rules([dict(H=4096, I=1024, E=512, k=10, t_min=1, t_max=256, nmax=16)])
        assert qb.forward_launches(qb.dims(4096, 10, 4096, 1024, 512), "mxfp4") == 6
        assert qb.forward_launches(qb.dims(1, 10, 4096, 1024, 512), "mxfp4") == 5
        assert qb.forward_launches(qb.dims(8192, 8, 4096, 1408, 64), "w8a8") == 7
        assert qb.forward_launches(qb.dims(8192, 8, 4096, 1408, 64), "w4a8") == 7
        assert qb.forward_launches(qb.dims(100, 8, 2048, 768, 128), "w4a16") == 6
        assert qb.forward_launches(qb.dims(0, 8, 2048, 768, 128), "w4a16") == 1
        assert qb.forward_launches(qb.dims(16, 2, 250, 128, 8), "mxfp4") == 0
    finally:
        qb.set_tile_rules(rules)


def test_host_checks_reject_before_launch(lib):
    d = qb.dims(16, 2, 256, 128, 8)
    null = None
    # null pointers and bad dims return QMOE_ERR_ARG without touching the GPU
    assert lib.qmoe_align_sort(ctypes.byref(d), null, null, null, null, null, null, null, 0, null) == -1
    assert lib.qmoe_combine(ctypes.byref(d), null, null, null, null, null) == -1
    bad = qb.dims(16, 2, 256, 100, 8)
    assert lib.qmoe_gemm2_w4a16(ctypes.byref(bad), null, null, null, null, null, null, 0, null) == -1
    assert lib.qmoe_quant_act_mxfp8(4, 48, null, null, null, null) == -1
    misaligned = ctypes.c_void_p(0x1000 + 4)
    ok = ctypes.c_void_p(0x1000)
    assert lib.qmoe_gemm1_swiglu_w4a16(ctypes.byref(d), misaligned, ok, ok, ok, ok, ok, 0, null) == -1
    # W4A16 pre-pack and tile helpers: bad K, null pointers, sizes from the stated layout
    assert lib.qmoe_prepack_int4_weights(128, 100, ok, ok, ok, null) == -1
    assert lib.qmoe_prepack_int4_weights(128, 128, null, ok, ok, null) == -1
    assert qb.int4_weights_packed_bytes(300, 4096) == 3 * 64 * 4608 + 3 * 128 * 4
    # x tiles: max_tiles = ceil(32/112) + 8 = 9 tiles, 4 K steps of 112 rows x 128 bytes, one factor per row
    assert qb.w4a16_x_tiles_bytes(d) == 9 * 4 * 112 * 128 + 9 * 112 * 4
    assert qb.w4a16_h_tiles_bytes(d) == 9 * 2 * 112 * 128 + 9 * 112 * 4 * 4
    assert qb.w4a16_h_tiles_bytes(qb.dims(16, 2, 256, 96, 8)) == 0
    assert qb.w4a16_h16_tiles_bytes(d) == 9 * 2 * 112 * 128 + 9 * 112 * 4
    assert lib.qmoe_w4a16_h_to_f16(ctypes.byref(d), null, ok, ok, ok, 1 << 20, null) == -1
    assert lib.qmoe_permute_x_f16(ctypes.byref(d), null, ok, ok, ok, ok, 1 << 20, null) == -1
    assert lib.qmoe_moe_forward(7, ctypes.byref(d), *([null] * 10), 0, null) == -1
    # MXFP4 scale pre-pack: bad K, null pointers
    assert lib.qmoe_prepack_mx_scales(128, 100, ok, ok, null) == -1
    assert lib.qmoe_prepack_mx_scales(128, 128, null, ok, null) == -1
    assert qb.mx_scales_packed_bytes(300, 4096) == 3 * 32 * 512
    # MXFP4 stage 1, gathering form: null or misaligned inputs, a short workspace, an unsupported
    # shape (H % 256) -- all refused on the host before any launch
    g1g = lambda dd, xq, xs, srt, ws_bytes: lib.qmoe_gemm1_swiglu_mxfp4_gather(
        ctypes.byref(dd), xq, xs, srt, ok, ok, ok, ok, ok, ok, ws_bytes, null)
    assert g1g(d, null, ok, ok, 1 << 30) == -1
    assert g1g(d, ok, misaligned, ok, 1 << 30) == -1
    assert g1g(d, ok, ok, null, 1 << 30) == -1
    assert g1g(d, ok, ok, ok, 0) == -1
    assert g1g(qb.dims(16, 2, 128, 128, 8), ok, ok, ok, 1 << 30) == -2


def test_w8a8_host_checks(lib):
    d = qb.dims(16, 2, 256, 128, 8)
    null = None
    ok = ctypes.c_void_p(0x1000)
    big = 1 << 30
    # W8A8 tiles: the W4A16 block layout (9 tiles, K/64 steps of 112 rows x 128 bytes), one fp32 scale per
    # row, one int32 step maximum per (112-row half, 128-element step)
    assert qb.w8a8_tiles_bytes(d, 256) == 9 * 4 * 112 * 128 + 9 * 112 * 4 + 9 * 1 * 2 * 4
    assert qb.w8a8_tiles_bytes(d, 128) == 9 * 2 * 112 * 128 + 9 * 112 * 4 + 9 * 1 * 1 * 4
    assert qb.w8a8_tiles_bytes(d, 96) == 0 and qb.w8a8_tiles_bytes(d, 192) == 0
    assert qb.w8a8_tiles_bytes(d, 16512) == 0
    # null pointers -> QMOE_ERR_ARG before any launch
    assert lib.qmoe_permute_quant_int8(ctypes.byref(d), null, ok, ok, ok, ok, big, null) == -1
    assert lib.qmoe_quant_tiles_int8_f32(ctypes.byref(d), ok, null, ok, ok, big, null) == -1
    assert lib.qmoe_gemm1_swiglu_w8a8(ctypes.byref(d), ok, null, ok, ok, ok, null, ok, ok, big, null) == -1
    assert lib.qmoe_gemm2_w8a8(ctypes.byref(d), ok, ok, ok, ok, null, null, ok, ok, big, null) == -1
    # a misaligned debug buffer
    odd = ctypes.c_void_p(0x1000 + 4)
    assert lib.qmoe_gemm2_w8a8(ctypes.byref(d), ok, ok, ok, ok, ok, odd, ok, ok, big, null) == -1
    # shapes outside the tensor-core tiles (H % 256, I % 128, K <= 16384) -> QMOE_ERR_UNSUPPORTED, no launch
    for bad in (qb.dims(16, 2, 384, 128, 8), qb.dims(16, 2, 256, 192, 8), qb.dims(16, 2, 256, 16512, 8)):
        assert lib.qmoe_gemm1_swiglu_w8a8(ctypes.byref(bad), ok, ok, ok, ok, ok, null, ok, ok, big, null) == -2
        assert lib.qmoe_gemm2_w8a8(ctypes.byref(bad), ok, ok, ok, ok, ok, null, ok, ok, big, null) == -2
    # W4A8 (int4 weights, the same activation tiles): the same host checks
    assert lib.qmoe_gemm1_swiglu_w4a8(ctypes.byref(d), ok, null, ok, ok, ok, null, ok, ok, big, null) == -1
    assert lib.qmoe_gemm2_w4a8(ctypes.byref(d), ok, ok, ok, ok, null, null, ok, ok, big, null) == -1
    assert lib.qmoe_gemm2_w4a8(ctypes.byref(d), ok, ok, ok, ok, ok, odd, ok, ok, big, null) == -1
    for bad in (qb.dims(16, 2, 384, 128, 8), qb.dims(16, 2, 256, 192, 8)):
        assert lib.qmoe_gemm1_swiglu_w4a8(ctypes.byref(bad), ok, ok, ok, ok, ok, null, ok, ok, big, null) == -2
        assert lib.qmoe_gemm2_w4a8(ctypes.byref(bad), ok, ok, ok, ok, ok, null, ok, ok, big, null) == -2


def test_tile_rules_host_only(lib):
    d = qb.dims(4096, 10, 4096, 1024, 512)
    small = qb.dims(1000, 10, 4096, 1024, 512)
    try:
        qb.set_tile_rules([])
        assert qb.tile_nmax(d) == 112 and qb.tile_nmax(qb.dims(8192, 10, 4096, 1024, 512)) == 224  # built-in rule
        # an exact-shape rule for one token bucket; first match wins; 0 = any
        qb.set_tile_rules([dict(H=4096, I=1024, E=512, k=10, t_min=4000, t_max=5000, nmax=224),
                           dict(H=0, I=0, E=512, k=0, t_min=0, t_max=10**9, nmax=112)])
        assert qb.tile_nmax(d) == 224 and qb.tile_nmax(small) == 112
        # buffer sizes follow the table
        assert qb.mx_tiles_bytes(d, 4096) == (40960 // 224 + 1 + 512) * 32 * (224 * 128 + 2 * 512)
        # bad rules are refused and leave the table as it was
        for bad in (dict(nmax=128), dict(nmax=112, t_min=5, t_max=4), dict(nmax=224, H=-1)):
            with pytest.raises(qb.QmoeError):
                qb.set_tile_rules([bad])
        assert qb.tile_nmax(d) == 224
    finally:
        qb.set_tile_rules([])
    assert qb.tile_nmax(d) == 112


def test_packaged_tile_table_parses():
    if not os.path.exists(qb.TILE_TABLE_PATH):
        pytest.skip("no tile table shipped")
    rules = qb.read_tile_table(qb.TILE_TABLE_PATH)
    assert rules and all(r["nmax"] in (16, 112, 224) and r["t_min"] <= r["t_max"] for r in rules)
