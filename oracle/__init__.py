"""CPU oracle for the FP8 W8A8 hot path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct statements of what the path computes, in C
(``oracle.c``) behind this ctypes wrapper.  Only the tests, the smoke check and
the benchmark's CPU-baseline leg may import it; the product library and its
Python binding never do, and the two share no code.

Every function takes and returns numpy arrays.  Sources are cited in
``oracle.c`` (page title plus section / table / equation).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u8, u16, i32, i64, u32, u64 = (ctypes.c_uint8, ctypes.c_uint16, ctypes.c_int32,
                                       ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64)
        P = ctypes.c_void_p
        sig = {
            "oracle_bf16_to_f32": (ctypes.c_float, [u16]),
            "oracle_e4m3_decode": (ctypes.c_double, [u8]),
            "oracle_e4m3_encode": (u8, [ctypes.c_float]),
            "oracle_e4m3_encode_bits": (u8, [ctypes.c_float]),
            "oracle_e4m3_cross_check": (i64, [u32, u64, P]),
            "oracle_e4m3_encode_patterns": (None, [u32, u64, P]),
            "oracle_e4m3_encode_array": (None, [P, i64, P]),
            "oracle_e4m3_decode_array": (None, [P, i64, P]),
            "oracle_scale_from_amax": (ctypes.c_float, [ctypes.c_float]),
            "oracle_quantize_value": (u8, [ctypes.c_float, ctypes.c_float]),
            "oracle_quantize_blocks": (ctypes.c_int, [P, i64, i64, i64, i64, P, P]),
            "oracle_quantize_blocks_mode": (ctypes.c_int, [P, i64, i64, i64, i64, ctypes.c_int, P, P]),
            "oracle_scale_pow2_from_amax": (ctypes.c_float, [ctypes.c_float]),
            "oracle_amax_bf16": (ctypes.c_float, [P, i64]),
            "oracle_quantize_with_scale": (None, [P, i64, ctypes.c_float, P]),
            "oracle_block_gemm": (ctypes.c_int, [P, P, P, P, i64, i64, i64, P, P]),
            "oracle_block_gemm_entries": (ctypes.c_int, [P, P, P, P, i64, P, P, i64, P, P]),
            "oracle_block_gemm_f32acc": (ctypes.c_int, [P, P, P, P, i64, i64, i64, P]),
            "oracle_grouped_gemm": (ctypes.c_int, [P, P, i64, P, P, i32, P, P, i64, i64, P, P]),
            "oracle_dequant_value": (ctypes.c_float, [u8, ctypes.c_float]),
            "oracle_dequantize_blocks": (ctypes.c_int, [P, P, i64, i64, i64, i64, P]),
            "oracle_quant_error": (ctypes.c_int, [P, P, P, i64, i64, i64, i64, i64, i64, P]),
            "oracle_decode_attention": (ctypes.c_int, [P, ctypes.c_float, P, ctypes.c_float, P,
                                                        ctypes.c_float, P, i64, i64, i64, i64, i64,
                                                        ctypes.c_double, P, P]),
            "oracle_prefill_attention": (ctypes.c_int, [P, ctypes.c_float, P, ctypes.c_float, P,
                                                         ctypes.c_float, i64, i64, i64, i64, i64,
                                                         ctypes.c_double, P, P]),
            "oracle_bf16_from_f64": (u16, [ctypes.c_double]),
            "oracle_bf16_from_f64_array": (None, [P, i64, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def cdiv(a, b):
    return (a + b - 1) // b


# ---- E4M3 codec -------------------------------------------------------------

def e4m3_decode(codes):
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    lib().oracle_e4m3_decode_array(_p(codes), codes.size, _p(out))
    return out


def e4m3_encode(x):
    """Encoder A (nearest-grid search) on a float32 array."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().oracle_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def e4m3_encode_bits_scalar(v):
    return lib().oracle_e4m3_encode_bits(float(v))


def e4m3_encode_scalar(v):
    return lib().oracle_e4m3_encode(float(v))


def e4m3_cross_check(start, count):
    """Mismatches between encoders A and B over bit patterns [start, start+count)."""
    first = np.zeros(1, np.uint32)
    bad = lib().oracle_e4m3_cross_check(start, count, _p(first))
    return int(bad), int(first[0])


def e4m3_encode_patterns(start, count):
    """Expected E4M3 code of every binary32 bit pattern in [start, start+count)."""
    out = np.empty(count, np.uint8)
    lib().oracle_e4m3_encode_patterns(start, count, _p(out))
    return out


# ---- quantizers -------------------------------------------------------------

def scale_from_amax(amax):
    return lib().oracle_scale_from_amax(float(amax))


def scale_pow2_from_amax(amax):
    return lib().oracle_scale_pow2_from_amax(float(amax))


def quantize_blocks(x_bf16_bits, br, bc, pow2=False):
    """x_bf16_bits: uint16 [rows, cols].  Returns (q uint8 [rows, cols],
    s float32 [ceil(rows/br), ceil(cols/bc)]).  pow2: power-of-two scales
    (NeMo blog, recipe variants), S = the smallest 2^e with 448 S >= amax."""
    x = _c(x_bf16_bits, np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((cdiv(rows, br), cdiv(cols, bc)), np.float32)
    rc = lib().oracle_quantize_blocks_mode(_p(x), rows, cols, br, bc, 1 if pow2 else 0, _p(q), _p(s))
    assert rc == 0
    return q, s


def quantize_weight_blockwise(w_bits):
    """Weights: 128x128 blocks."""
    return quantize_blocks(w_bits, 128, 128)


def quantize_act_per_token_group(x_bits):
    """Activations: 1x128 per-token groups."""
    return quantize_blocks(x_bits, 1, 128)


def quantize_act_per_token_group_gather(x_bits, row_idx):
    """Routed rows (FP8-RL page, section 1: the expert layers' inputs): row r
    of the result is the 1x128 group quantization of x row row_idx[r]; an
    index outside [0, rows_x) stands for an all-zero row.  Gather first
    (numpy indexing), then the block quantizer."""
    x = _c(x_bits, np.uint16)
    ri = np.asarray(row_idx, dtype=np.int64).reshape(-1)
    rows_x, k = x.shape
    g = np.zeros((ri.size, k), np.uint16)
    ok = (ri >= 0) & (ri < rows_x)
    g[ok] = x[ri[ok]]
    return quantize_blocks(g, 1, 128)


def dequantize_blocks(q, s, br, bc):
    """Fake quant ([UFP8] quantize-dequantize experiments): BF16 bits of
    dec(q) * S (one binary32 multiply, then BF16 round to nearest even)."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    rows, cols = q.shape
    y = np.empty((rows, cols), np.uint16)
    assert lib().oracle_dequantize_blocks(_p(q), _p(s), rows, cols, br, bc, _p(y)) == 0
    return y


def quant_error(x_bits, q, s, sbr, sbc, rbr, rbc):
    """Per report block (rbr x rbc): [max |x - x_hat|, sum (x - x_hat)^2,
    sum x^2] in FP64, x_hat = dec(q) * S in binary32; shape
    [ceil(rows/rbr), ceil(cols/rbc), 3]."""
    x = _c(x_bits, np.uint16)
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    rows, cols = x.shape
    st = np.empty((cdiv(rows, rbr), cdiv(cols, rbc), 3), np.float64)
    assert lib().oracle_quant_error(_p(x), _p(q), _p(s), rows, cols, sbr, sbc, rbr, rbc,
                                    _p(st)) == 0
    return st


def amax_bf16(x_bits):
    x = _c(x_bits, np.uint16).reshape(-1)
    return lib().oracle_amax_bf16(_p(x), x.size)


def quantize_with_scale(x_bits, scale):
    x = _c(x_bits, np.uint16)
    q = np.empty(x.shape, np.uint8)
    lib().oracle_quantize_with_scale(_p(x), x.size, float(scale), _p(q))
    return q


def kv_amax_quantize(x_bits):
    """Per-tensor: amax over the whole tensor, one scale, every element coded.
    Returns (q, scale, amax)."""
    x = _c(x_bits, np.uint16)
    flat = x.reshape(1, -1)
    n = flat.shape[1]
    q = np.empty(flat.shape, np.uint8)
    s = np.empty((1, 1), np.float32)
    if n:
        rc = lib().oracle_quantize_blocks(_p(flat), 1, n, 1, n, _p(q), _p(s))
        assert rc == 0
    else:
        s[0, 0] = 1.0
    return q.reshape(x.shape), float(s[0, 0]), amax_bf16(x)


# ---- GEMMs -----------------------------------------------------------------

def block_gemm(xq, xs, wq, ws):
    """Y = X W^T with blockwise scales.  Returns (y float64 [m,n], absref [m,n])."""
    xq, xs, wq, ws = _c(xq, np.uint8), _c(xs, np.float32), _c(wq, np.uint8), _c(ws, np.float32)
    m, k = xq.shape
    n = wq.shape[0]
    y = np.empty((m, n), np.float64)
    a = np.empty((m, n), np.float64)
    rc = lib().oracle_block_gemm(_p(xq), _p(xs), _p(wq), _p(ws), m, n, k, _p(y), _p(a))
    assert rc == 0
    return y, a


def block_gemm_entries(xq, xs, wq, ws, ii, jj):
    xq, xs, wq, ws = _c(xq, np.uint8), _c(xs, np.float32), _c(wq, np.uint8), _c(ws, np.float32)
    ii, jj = _c(ii, np.int64), _c(jj, np.int64)
    k = xq.shape[1]
    y = np.empty(ii.shape, np.float64)
    a = np.empty(ii.shape, np.float64)
    lib().oracle_block_gemm_entries(_p(xq), _p(xs), _p(wq), _p(ws), k, _p(ii), _p(jj),
                                    ii.size, _p(y), _p(a))
    return y, a


def block_gemm_f32acc(xq, xs, wq, ws):
    xq, xs, wq, ws = _c(xq, np.uint8), _c(xs, np.float32), _c(wq, np.uint8), _c(ws, np.float32)
    m, k = xq.shape
    n = wq.shape[0]
    y = np.empty((m, n), np.float32)
    lib().oracle_block_gemm_f32acc(_p(xq), _p(xs), _p(wq), _p(ws), m, n, k, _p(y))
    return y


def grouped_gemm(xq, xs, row_idx, group_offsets, wq, ws):
    """wq [g, n, k], ws [g, ceil(n/128), ceil(k/128)]; row_idx may be None."""
    xq, xs, wq, ws = _c(xq, np.uint8), _c(xs, np.float32), _c(wq, np.uint8), _c(ws, np.float32)
    off = _c(group_offsets, np.int32)
    ri = None if row_idx is None else _c(row_idx, np.int32)
    g, n, k = wq.shape
    total = int(off[-1])
    y = np.empty((total, n), np.float64)
    a = np.empty((total, n), np.float64)
    rc = lib().oracle_grouped_gemm(_p(xq), _p(xs), xq.shape[0], _p(ri), _p(off), g,
                                   _p(wq), _p(ws), n, k, _p(y), _p(a))
    assert rc == 0
    return y, a


def decode_attention(q, sq, k, sk, v, sv, lens, softmax_scale):
    """FP8 decode attention (NeMo blog Table 3, per-tensor Q/K/V scales):
    q [B, Hq, D], k and v [B, S, Hkv, D] E4M3 codes, lens [B].  Returns
    (out, absout) float64 [B, Hq, D]: the exact-math output and the bound
    sv * sum_t p_t |dec(v_t)| used for its tolerance."""
    q, k, v = _c(q, np.uint8), _c(k, np.uint8), _c(v, np.uint8)
    lens = _c(lens, np.int32)
    B, Hq, D = q.shape
    S, Hkv = k.shape[1], k.shape[2]
    out = np.empty((B, Hq, D), np.float64)
    ab = np.empty((B, Hq, D), np.float64)
    rc = lib().oracle_decode_attention(_p(q), float(sq), _p(k), float(sk), _p(v), float(sv), _p(lens),
                                       B, S, Hq, Hkv, D, float(softmax_scale), _p(out), _p(ab))
    assert rc == 0
    return out, ab


def prefill_attention(q, sq, k, sk, v, sv, softmax_scale):
    """Causal prefill attention over FP8 Q, K, V (NeMo blog Table 3, per-tensor
    scales): q [B, S, Hq, D], k and v [B, S, Hkv, D] E4M3 codes; query token i
    reads tokens 0..i.  Returns (out, absout) float64 [B, S, Hq, D]: the
    exact-math output and the bound sv * sum_j p_j |dec(v_j)| for its
    tolerance."""
    q, k, v = _c(q, np.uint8), _c(k, np.uint8), _c(v, np.uint8)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    out = np.empty((B, S, Hq, D), np.float64)
    ab = np.empty((B, S, Hq, D), np.float64)
    rc = lib().oracle_prefill_attention(_p(q), float(sq), _p(k), float(sk), _p(v), float(sv),
                                        B, S, Hq, Hkv, D, float(softmax_scale), _p(out), _p(ab))
    assert rc == 0
    return out, ab


def bf16_from_f64(y):
    y = _c(y, np.float64)
    out = np.empty(y.shape, np.uint16)
    lib().oracle_bf16_from_f64_array(_p(y), y.size, _p(out))
    return out


def bf16_bits_to_f64(b):
    b = _c(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
