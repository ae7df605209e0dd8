"""CPU-side checks of the C ABI: the library builds, loads without a GPU and
exports every function include/w8a8fp8.h declares, and bad arguments are
rejected on the host with the documented status before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w8a8fp8.h")


@pytest.fixture(scope="module")
def L():
    from w8a8_gemm_rl_gb300 import _build
    _build.build()
    import w8a8_gemm_rl_gb300 as W
    return W.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_hot_path_calls():
    names = _declared_functions()
    for n in ["quantize_weight_blockwise", "quantize_act_per_token_group", "fp8_block_gemm",
              "fp8_grouped_gemm", "kv_amax_quantize", "e4m3_encode_f32", "e4m3_decode_f32"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    assert L.w8a8_version() == 200
    for s in range(6):
        assert L.w8a8_status_string(s)
    assert L.w8a8_status_string(0) == b"ok"


OK, NULL, SHAPE, ALIGN, UNSUP = 0, 1, 2, 3, 4
A = 0x10000  # a fake, 16-byte aligned "device" address: never dereferenced on these paths


def test_quantizer_argument_checks(L):
    q = L.quantize_act_per_token_group
    assert q(None, 4, 128, A, A, None) == NULL
    assert q(A, -1, 128, A, A, None) == SHAPE
    assert q(A, 4, -5, A, A, None) == SHAPE
    assert q(A + 2, 4, 128, A, A, None) == ALIGN
    assert q(A, 4, 128, A + 8, A, None) == ALIGN
    assert q(A, 4, 128, A, A + 2, None) == ALIGN
    assert q(None, 0, 128, None, None, None) == OK  # empty: nothing to do
    assert q(None, 4, 0, None, None, None) == OK
    w = L.quantize_weight_blockwise
    assert w(A, 256, 128, None, A, None) == NULL
    assert w(A, 256, 128, A, None, None) == NULL
    assert w(A + 4, 256, 128, A, A, None) == ALIGN
    assert w(None, 0, 0, None, None, None) == OK
    b = L.quantize_weight_blockwise_batched
    assert b(None, 3, None) == NULL
    assert b(None, -1, None) == SHAPE
    assert b(None, 0, None) == OK
    import w8a8_gemm_rl_gb300 as W
    descs = (W.WeightDesc * 2)(W.WeightDesc(A, A, A, 128, 128), W.WeightDesc(A, None, A, 128, 128))
    assert b(ctypes.cast(descs, ctypes.c_void_p), 2, None) == NULL


def test_gather_quantizer_argument_checks(L):
    g = L.quantize_act_per_token_group_gather
    assert g(A, -1, 128, A, 5, A, A, None) == SHAPE
    assert g(A, 10, -2, A, 5, A, A, None) == SHAPE
    assert g(A, 10, 128, A, -5, A, A, None) == SHAPE
    assert g(None, 10, 128, None, 0, None, None, None) == OK  # nothing routed
    assert g(A, 10, 0, A, 5, A, A, None) == OK  # empty rows
    assert g(A, 10, 128, None, 5, A, A, None) == NULL
    assert g(None, 10, 128, A, 5, A, A, None) == NULL
    assert g(A, 10, 128, A, 5, None, A, None) == NULL
    assert g(A + 2, 10, 128, A, 5, A, A, None) == ALIGN
    assert g(A, 10, 128, A + 2, 5, A, A, None) == ALIGN
    assert g(A, 10, 128, A, 5, A + 8, A, None) == ALIGN
    assert g(A, 10, 100, A, 5, A, A, None) == UNSUP  # k % 8


def test_dequant_and_report_argument_checks(L):
    d = L.dequantize_blockwise
    assert d(A, A, -1, 128, 1, 128, A, None) == SHAPE
    assert d(A, A, 4, 128, 0, 128, A, None) == SHAPE
    assert d(None, None, 0, 128, 1, 128, None, None) == OK
    assert d(None, A, 4, 128, 1, 128, A, None) == NULL
    assert d(A, A, 4, 128, 1, 128, A + 2, None) == ALIGN
    assert d(A + 8, A, 4, 128, 1, 128, A, None) == ALIGN
    r = L.quant_error_report
    assert r(A, A, A, 4, 128, 1, 0, 1, 128, A, None) == SHAPE
    assert r(A, A, A, 4, 128, 1, 128, -1, 128, A, None) == SHAPE
    assert r(A, A, A, 4, 128, 1, 128, 1, 128, None, None) == NULL
    assert r(A, A, A, 4, 128, 1, 128, 1, 128, A + 4, None) == ALIGN
    assert r(A + 2, A, A, 4, 128, 1, 128, 1, 128, A, None) == ALIGN
    assert r(A, A, A, 4, 1 << 21, 1, 128, 1, 1 << 21, A, None) == UNSUP
    assert r(None, None, None, 0, 128, 1, 128, 1, 128, None, None) == OK


def test_pow2_quantizer_argument_checks(L):
    for f in (L.quantize_weight_blockwise_pow2, L.quantize_act_per_token_group_pow2):
        assert f(None, 4, 128, A, A, None) == NULL
        assert f(A, -1, 128, A, A, None) == SHAPE
        assert f(A + 2, 4, 128, A, A, None) == ALIGN
        assert f(None, 0, 128, None, None, None) == OK


def test_attention_argument_checks(L):
    import ctypes
    a = L.fp8_decode_attention
    sc = ctypes.c_float(0.088)
    assert a(A, A, A, A, A, A, A, 2, 64, 8, 2, 64, sc, A, None) == UNSUP    # head dim
    assert a(A, A, A, A, A, A, A, 2, 64, 12, 4, 128, sc, A, None) == UNSUP  # group of 3
    assert a(A, A, A, A, A, A, A, 2, 64, 8, 3, 128, sc, A, None) == SHAPE   # 8 % 3
    assert a(A, A, A, A, A, A, A, -1, 64, 8, 2, 128, sc, A, None) == SHAPE
    assert a(None, None, None, None, None, None, None, 0, 64, 8, 2, 128, sc, None, None) == OK
    assert a(A, A, None, A, A, A, A, 2, 64, 8, 2, 128, sc, A, None) == NULL
    assert a(A, A, A + 4, A, A, A, A, 2, 64, 8, 2, 128, sc, A, None) == ALIGN
    assert a(A, A, A, A, A, A, A, 2, 64, 8, 2, 128, sc, A + 2, None) == ALIGN
    # TMA row coordinates are 32-bit: batch * max_seq must stay below 2^31 - 32
    assert a(A, A, A, A, A, A, A, 1 << 16, 1 << 15, 8, 2, 128, sc, A, None) == UNSUP
    assert a(A, A, A, A, A, A, A, 1 << 31, 1, 8, 2, 128, sc, A, None) == UNSUP
    assert a(A, A, A, A, A, A, A, 1, 1 << 31, 8, 2, 128, sc, A, None) == UNSUP


def test_prefill_attention_argument_checks(L):
    import ctypes
    a = L.fp8_prefill_attention
    sc = ctypes.c_float(0.088)
    assert a(A, A, A, A, A, A, 2, 64, 8, 2, 64, sc, A, None) == UNSUP    # head dim
    assert a(A, A, A, A, A, A, 2, 64, 8, 3, 128, sc, A, None) == SHAPE   # 8 % 3
    assert a(A, A, A, A, A, A, -1, 64, 8, 2, 128, sc, A, None) == SHAPE
    assert a(A, A, A, A, A, A, 2, -5, 8, 2, 128, sc, A, None) == SHAPE
    assert a(None, None, None, None, None, None, 0, 64, 8, 2, 128, sc, None, None) == OK
    assert a(None, None, None, None, None, None, 3, 0, 8, 2, 128, sc, None, None) == OK
    assert a(A, A, None, A, A, A, 2, 64, 8, 2, 128, sc, A, None) == NULL
    assert a(A, A, A + 4, A, A, A, 2, 64, 8, 2, 128, sc, A, None) == ALIGN
    assert a(A, A, A, A, A, A, 2, 64, 8, 2, 128, sc, A + 2, None) == ALIGN
    assert a(A, A, A, A, A, A, 2, 64, 8, 2, 128, sc, A + 8, None) == ALIGN  # out: 16 bytes
    # grid limits and 32-bit TMA row coordinates
    assert a(A, A, A, A, A, A, 1 << 16, 1, 8, 2, 128, sc, A, None) == UNSUP
    assert a(A, A, A, A, A, A, 2, 64, 1 << 16, 2, 128, sc, A, None) == UNSUP
    assert a(A, A, A, A, A, A, 1 << 15, 1 << 16, 8, 2, 128, sc, A, None) == UNSUP
    # the last key tile of the last sequence starts below 2^31 - 128
    assert a(A, A, A, A, A, A, 2, (1 << 30) - 63, 8, 2, 128, sc, A, None) == UNSUP


def test_gemm_argument_checks(L):
    g = L.fp8_block_gemm
    assert g(A, A, A, A, A, 128, 256, 100, None) == SHAPE  # k % 16
    assert g(A, A, A, A, A, 128, 252, 128, None) == SHAPE  # n % 8
    assert g(A, A, A, A, A, -1, 256, 128, None) == SHAPE
    assert g(A, A, A, A, None, 128, 256, 128, None) == NULL
    assert g(None, A, A, A, A, 128, 256, 128, None) == NULL
    assert g(A + 1, A, A, A, A, 128, 256, 128, None) == ALIGN
    assert g(A, A + 1, A, A, A, 128, 256, 128, None) == ALIGN
    assert g(A, A, A, A, A + 8, 128, 256, 128, None) == ALIGN
    assert g(None, None, None, None, None, 0, 256, 128, None) == OK
    assert g(A, A, A, A, A, 1 << 31, 256, 128, None) == SHAPE
    li = L.w8a8_linear
    assert li(A, 64, 100, A, A, 256, A, None, None, 0, None) == SHAPE   # k % 16
    assert li(A, 64, 128, A, A, 256, A, A, None, 0, None) == NULL       # xq without xs
    assert li(A, 300, 128, A, A, 256, A, None, None, 0, None) == NULL   # m > 128 needs xq, xs
    assert li(A + 2, 64, 128, A, A, 256, A, None, None, 0, None) == ALIGN
    assert li(A, 64, 128, A, A, 2048, A, None, None, 0, None) == NULL   # wide n: two kernels
    assert li(A, 64, 128, A, A, 256, A, None, None, 4, None) == UNSUP
    assert li(None, 0, 128, None, None, 256, None, None, None, 0, None) == OK
    ge = L.fp8_block_gemm_ex
    assert ge(A, A, A, A, A, 128, 256, 100, 0, None) == SHAPE
    assert ge(A, A, A, A, A + 8, 64, 256, 128, 1, None) == ALIGN
    assert ge(A, A, A, A, A, 64, 256, 128, 2, None) == UNSUP  # unknown flag bit
    assert ge(None, None, None, None, None, 0, 256, 128, 1, None) == OK
    gg = L.fp8_grouped_gemm
    assert gg(A, A, 10, None, A, 2, 11, A, A, A, 256, 128, None) == SHAPE  # identity reads past rows_x
    assert gg(A, A, 10, None, None, 2, 10, A, A, A, 256, 128, None) == NULL
    assert gg(A, A, 10, A + 2, A, 2, 10, A, A, A, 256, 128, None) == ALIGN
    assert gg(A, A, 10, A, A, -1, 10, A, A, A, 256, 128, None) == SHAPE
    assert gg(A, A, 10, A, A, 100000, 10, A, A, A, 256, 128, None) == UNSUP
    assert gg(A, A, 10, A, A, 2, 10, A, A, A, 256, 120, None) == SHAPE
    assert gg(None, None, 0, None, None, 0, 0, None, None, None, 256, 128, None) == OK


def test_kv_and_codec_argument_checks(L):
    kv = L.kv_amax_quantize
    assert kv(A, 100, A, A, A, 7, None) == UNSUP
    assert kv(A, 100, A, None, A, 0, None) == NULL
    assert kv(A, 100, A, A, None, 0, None) == NULL
    assert kv(A, 100, None, A, A, 0, None) == NULL
    assert kv(A + 2, 100, A, A, A, 0, None) == ALIGN
    assert kv(A, -1, A, A, A, 0, None) == SHAPE
    assert L.e4m3_encode_f32(None, 10, A, None) == NULL
    assert L.e4m3_encode_f32(A + 4, 10, A, None) == ALIGN
    assert L.e4m3_decode_f32(A, -1, A, None) == SHAPE
    assert L.e4m3_decode_f32(None, 0, None, None) == OK
