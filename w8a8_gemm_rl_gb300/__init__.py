"""Python binding of the GB300 FP8 W8A8 library (libw8a8fp8.so).

Argument marshalling only: each function checks the tensors it is given,
allocates outputs with torch when the caller passes none, and calls the C
entry point of the same name on the current CUDA stream.  Every step of the
computation runs in the library's CUDA kernels; there is no other code path,
and a missing library is an error.

The C ABI and what each call computes are documented in include/w8a8fp8.h.
"""
import ctypes
import math
import os

import torch

__all__ = [
    "lib", "W8A8Error", "e4m3_encode_f32", "e4m3_decode_f32", "quantize_weight_blockwise",
    "quantize_weight_blockwise_batched", "quantize_act_per_token_group",
    "quantize_act_per_token_group_gather", "dequantize_blockwise", "quant_error_report",
    "sqnr_db", "fp8_decode_attention", "fp8_prefill_attention", "dequantize_blockwise_batched", "quant_error_report_batched",
    "fp8_block_gemm", "fp8_block_gemm_pow2",
    "fp8_grouped_gemm", "kv_amax_quantize", "w8a8_linear", "consume_device_error",
    "GEMM_STATIC_WEIGHTS", "LINEAR_SINGLE_KERNEL", "debug_force_wait_timeout",
    "KV_AMAX_AND_QUANT", "KV_AMAX_ONLY", "KV_QUANT_ONLY", "LIB_PATH",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libw8a8fp8.so")

KV_AMAX_AND_QUANT, KV_AMAX_ONLY, KV_QUANT_ONLY = 0, 1, 2


class W8A8Error(RuntimeError):
    def __init__(self, name, status, msg, cuda_msg=""):
        super().__init__(f"{name}: status {status} ({msg})" + (f": {cuda_msg}" if cuda_msg else ""))
        self.status = status


class WeightDesc(ctypes.Structure):
    _fields_ = [("w_bf16", ctypes.c_void_p), ("wq", ctypes.c_void_p), ("ws", ctypes.c_void_p),
                ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


_lib = None

_P, _I64, _I32, _INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
_SIGNATURES = {
    "w8a8_status_string": (ctypes.c_char_p, [_INT]),
    "w8a8_version": (_INT, []),
    "w8a8_last_cuda_error": (ctypes.c_char_p, []),
    "w8a8_consume_device_error": (_INT, [_P]),
    "w8a8_debug_force_wait_timeout": (_INT, [_INT]),
    "e4m3_encode_f32": (_INT, [_P, _I64, _P, _P]),
    "e4m3_decode_f32": (_INT, [_P, _I64, _P, _P]),
    "quantize_weight_blockwise": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "quantize_weight_blockwise_batched": (_INT, [_P, _I32, _P]),
    "quantize_weight_blockwise_batched_pow2": (_INT, [_P, _I32, _P]),
    "quantize_act_per_token_group": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "quantize_weight_blockwise_pow2": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "quantize_act_per_token_group_pow2": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "quantize_act_per_token_group_gather": (_INT, [_P, _I64, _I64, _P, _I64, _P, _P, _P]),
    "dequantize_blockwise": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _P, _P]),
    "quant_error_report": (_INT, [_P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _P, _P]),
    "fp8_decode_attention": (_INT, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32,
                                    ctypes.c_float, _P, _P]),
    "fp8_prefill_attention": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32,
                                     ctypes.c_float, _P, _P]),
    "fp8_block_gemm": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "fp8_block_gemm_ex": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_uint32, _P]),
    "fp8_block_gemm_pow2": (_INT, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w8a8_linear": (_INT, [_P, _I64, _I64, _P, _P, _I64, _P, _P, _P, ctypes.c_uint32, _P]),
    "fp8_grouped_gemm": (_INT, [_P, _P, _I64, _P, _P, _I32, _I64, _P, _P, _P, _I64, _I64, _P]),
    "kv_amax_quantize": (_INT, [_P, _I64, _P, _P, _P, _INT, _P]),
    "dequantize_blockwise_batched": (_INT, [_P, _I32, _P]),
    "quant_error_report_batched": (_INT, [_P, _I32, _P]),
}


def lib():
    """The loaded C library (ctypes), with argument types declared."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with w8a8_gemm_rl_gb300._build.build() "
                "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(name, status):
    if status != 0:
        L = lib()
        raise W8A8Error(name, status, L.w8a8_status_string(status).decode(),
                        L.w8a8_last_cuda_error().decode() if status == 5 else "")


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")


def _cdiv(a, b):
    return (a + b - 1) // b


# ------------------------------------------------------------------ codec

def e4m3_encode_f32(x, out=None, stream=None):
    _need(x, torch.float32, "x")
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if out is None else out
    _check("e4m3_encode_f32", lib().e4m3_encode_f32(_ptr(x), x.numel(), _ptr(q), _stream(stream)))
    return q


def e4m3_decode_f32(q, out=None, stream=None):
    _need(q, torch.uint8, "q")
    x = torch.empty(q.shape, dtype=torch.float32, device=q.device) if out is None else out
    _check("e4m3_decode_f32", lib().e4m3_decode_f32(_ptr(q), q.numel(), _ptr(x), _stream(stream)))
    return x


# ------------------------------------------------------------- quantizers

def quantize_weight_blockwise(w, wq=None, ws=None, stream=None, pow2=False):
    """w BF16 [n, k] -> (wq uint8 [n, k], ws float32 [ceil(n/128), ceil(k/128)]);
    pow2: power-of-two scales (quantize_weight_blockwise_pow2)."""
    _need(w, torch.bfloat16, "w")
    n, k = w.shape
    wq = torch.empty((n, k), dtype=torch.uint8, device=w.device) if wq is None else wq
    ws = torch.empty((_cdiv(n, 128), _cdiv(k, 128)), dtype=torch.float32, device=w.device) if ws is None else ws
    name = "quantize_weight_blockwise_pow2" if pow2 else "quantize_weight_blockwise"
    _check(name, getattr(lib(), name)(_ptr(w), n, k, _ptr(wq), _ptr(ws), _stream(stream)))
    return wq, ws


def quantize_weight_blockwise_batched(ws_in, outs=None, stream=None, pow2=False):
    """Quantize a list of BF16 weight matrices in one call.  Returns a list of
    (wq, ws) pairs (or fills `outs`, a list of such pairs).  pow2:
    power-of-two scales."""
    if outs is None:
        outs = []
        for w in ws_in:
            n, k = w.shape
            outs.append((torch.empty((n, k), dtype=torch.uint8, device=w.device),
                         torch.empty((_cdiv(n, 128), _cdiv(k, 128)), dtype=torch.float32, device=w.device)))
    descs = (WeightDesc * len(ws_in))()
    for i, (w, (q, s)) in enumerate(zip(ws_in, outs)):
        _need(w, torch.bfloat16, "w")
        descs[i] = WeightDesc(w.data_ptr(), q.data_ptr(), s.data_ptr(), w.shape[0], w.shape[1])
    name = "quantize_weight_blockwise_batched_pow2" if pow2 else "quantize_weight_blockwise_batched"
    _check(name, getattr(lib(), name)(ctypes.cast(descs, ctypes.c_void_p), len(ws_in), _stream(stream)))
    return outs


def quantize_act_per_token_group(x, xq=None, xs=None, stream=None, pow2=False):
    """x BF16 [m, k] -> (xq uint8 [m, k], xs float32 [m, ceil(k/128)]);
    pow2: power-of-two scales (quantize_act_per_token_group_pow2)."""
    _need(x, torch.bfloat16, "x")
    m, k = x.shape
    xq = torch.empty((m, k), dtype=torch.uint8, device=x.device) if xq is None else xq
    xs = torch.empty((m, _cdiv(k, 128)), dtype=torch.float32, device=x.device) if xs is None else xs
    name = "quantize_act_per_token_group_pow2" if pow2 else "quantize_act_per_token_group"
    _check(name, getattr(lib(), name)(_ptr(x), m, k, _ptr(xq), _ptr(xs), _stream(stream)))
    return xq, xs


def quantize_act_per_token_group_gather(x, row_idx, xq=None, xs=None, stream=None):
    """x BF16 [rows_x, k], row_idx int32 [total] -> (xq uint8 [total, k],
    xs float32 [total, ceil(k/128)]): row r quantizes x[row_idx[r]]."""
    _need(x, torch.bfloat16, "x")
    _need(row_idx, torch.int32, "row_idx")
    rows_x, k = x.shape
    total = row_idx.shape[0]
    xq = torch.empty((total, k), dtype=torch.uint8, device=x.device) if xq is None else xq
    xs = torch.empty((total, _cdiv(k, 128)), dtype=torch.float32, device=x.device) if xs is None else xs
    _check("quantize_act_per_token_group_gather",
           lib().quantize_act_per_token_group_gather(_ptr(x), rows_x, k, _ptr(row_idx), total,
                                                     _ptr(xq), _ptr(xs), _stream(stream)))
    return xq, xs


def dequantize_blockwise(q, s, block_rows, block_cols, y=None, stream=None):
    """q uint8 [rows, cols], s float32 scale grid -> BF16 [rows, cols] of dec(q) * S."""
    _need(q, torch.uint8, "q")
    rows, cols = q.shape
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=q.device) if y is None else y
    _check("dequantize_blockwise",
           lib().dequantize_blockwise(_ptr(q), _ptr(s), rows, cols, block_rows, block_cols,
                                      _ptr(y), _stream(stream)))
    return y


def quant_error_report(x, q, s, scale_block, report_block, stats=None, stream=None):
    """Per report block: float64 [..., 3] = (max |x - x_hat|, sum e^2, sum x^2)."""
    _need(x, torch.bfloat16, "x")
    _need(q, torch.uint8, "q")
    rows, cols = x.shape
    rbr, rbc = report_block
    if stats is None:
        stats = torch.empty((_cdiv(rows, rbr), _cdiv(cols, rbc), 3), dtype=torch.float64,
                            device=x.device)
    _check("quant_error_report",
           lib().quant_error_report(_ptr(x), _ptr(q), _ptr(s), rows, cols, scale_block[0],
                                    scale_block[1], rbr, rbc, _ptr(stats), _stream(stream)))
    return stats


class DequantDesc(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("y_bf16", ctypes.c_void_p),
                ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


class ErrorDesc(ctypes.Structure):
    _fields_ = [("x_bf16", ctypes.c_void_p), ("q", ctypes.c_void_p), ("s", ctypes.c_void_p),
                ("stats", ctypes.c_void_p), ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


def dequantize_blockwise_batched(qs, ss, ys=None, stream=None):
    """dequantize_blockwise over many matrices with 128 x 128 scale blocks in
    one call: qs uint8 [n, k] codes, ss their scale grids; returns the BF16
    outputs (allocated unless ys is given)."""
    if ys is None:
        ys = [torch.empty(q.shape, dtype=torch.bfloat16, device=q.device) for q in qs]
    arr = (DequantDesc * len(qs))()
    for i, (q, s, y) in enumerate(zip(qs, ss, ys)):
        _need(q, torch.uint8, "q")
        arr[i] = DequantDesc(q.data_ptr(), s.data_ptr(), y.data_ptr(), q.shape[0], q.shape[1])
    _check("dequantize_blockwise_batched",
           lib().dequantize_blockwise_batched(arr, len(qs), _stream(stream)))
    return ys


def quant_error_report_batched(xs, qs, ss, stats=None, stream=None):
    """quant_error_report over many matrices with 128 x 128 scale and report
    blocks in one call; returns the float64 [ceil(n/128), ceil(k/128), 3]
    reports (allocated unless stats is given)."""
    if stats is None:
        stats = [torch.empty((_cdiv(x.shape[0], 128), _cdiv(x.shape[1], 128), 3),
                             dtype=torch.float64, device=x.device) for x in xs]
    arr = (ErrorDesc * len(xs))()
    for i, (x, q, s, st) in enumerate(zip(xs, qs, ss, stats)):
        _need(x, torch.bfloat16, "x")
        _need(q, torch.uint8, "q")
        arr[i] = ErrorDesc(x.data_ptr(), q.data_ptr(), s.data_ptr(), st.data_ptr(), x.shape[0],
                           x.shape[1])
    _check("quant_error_report_batched",
           lib().quant_error_report_batched(arr, len(xs), _stream(stream)))
    return stats


def sqnr_db(stats):
    """10 log10(sum x^2 / sum e^2) over all blocks of a report."""
    import math
    se = float(stats[..., 1].sum())
    sx = float(stats[..., 2].sum())
    return math.inf if se == 0.0 else 10.0 * math.log10(sx / se)


def fp8_decode_attention(q, q_scale, k_cache, k_scale, v_cache, v_scale, seq_lens,
                         softmax_scale=None, out=None, stream=None):
    """Decode attention over the FP8 KV cache (one query token per sequence).

    q uint8 [B, Hq, 128] E4M3 codes; k_cache, v_cache uint8 [B, S, Hkv, 128];
    q_scale, k_scale, v_scale float32 [1] per-tensor scales (device); seq_lens
    int32 [B] (device; clamped to [0, S] by the kernel) -> BF16 [B, Hq, 128].
    Query head h reads KV head h // (Hq // Hkv); softmax_scale defaults to
    1/sqrt(128)."""
    _need(q, torch.uint8, "q")
    _need(k_cache, torch.uint8, "k_cache")
    _need(v_cache, torch.uint8, "v_cache")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, D = q.shape
    S, Hkv = k_cache.shape[1], k_cache.shape[2]
    sc = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device) if out is None else out
    _check("fp8_decode_attention",
           lib().fp8_decode_attention(_ptr(q), _ptr(q_scale), _ptr(k_cache), _ptr(k_scale),
                                      _ptr(v_cache), _ptr(v_scale), _ptr(seq_lens), B, S, Hq, Hkv,
                                      D, sc, _ptr(out), _stream(stream)))
    return out


def fp8_prefill_attention(q, q_scale, k, k_scale, v, v_scale, softmax_scale=None, out=None,
                          stream=None):
    """Causal prefill attention over FP8 Q, K and V.

    q uint8 [B, S, Hq, 128] E4M3 codes; k, v uint8 [B, S, Hkv, 128]; q_scale,
    k_scale, v_scale float32 [1] per-tensor scales (device) -> BF16
    [B, S, Hq, 128].  Query token i reads tokens 0..i of its sequence; query
    head h reads KV head h // (Hq // Hkv); softmax_scale defaults to
    1/sqrt(128)."""
    _need(q, torch.uint8, "q")
    _need(k, torch.uint8, "k")
    _need(v, torch.uint8, "v")
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    sc = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    out = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device=q.device) if out is None else out
    _check("fp8_prefill_attention",
           lib().fp8_prefill_attention(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(v),
                                       _ptr(v_scale), B, S, Hq, Hkv, D, sc, _ptr(out),
                                       _stream(stream)))
    return out


# ------------------------------------------------------------------ GEMMs

GEMM_STATIC_WEIGHTS = 1


def fp8_block_gemm(xq, xs, wq, ws, y=None, stream=None, static_weights=False):
    """Y = X W^T with blockwise FP32 scales; returns BF16 [m, n].
    static_weights: the caller states that wq and ws are not written by the
    kernel enqueued just before on the stream (fp8_block_gemm_ex's
    W8A8_GEMM_STATIC_WEIGHTS); the result is the same either way."""
    _need(xq, torch.uint8, "xq")
    _need(wq, torch.uint8, "wq")
    m, k = xq.shape
    n = wq.shape[0]
    y = torch.empty((m, n), dtype=torch.bfloat16, device=xq.device) if y is None else y
    if static_weights:
        _check("fp8_block_gemm_ex",
               lib().fp8_block_gemm_ex(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), _ptr(y), m, n, k,
                                       GEMM_STATIC_WEIGHTS, _stream(stream)))
    else:
        _check("fp8_block_gemm", lib().fp8_block_gemm(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws),
                                                      _ptr(y), m, n, k, _stream(stream)))
    return y


def fp8_block_gemm_pow2(xq, xs, wq, ws, y=None, stream=None):
    """Y = X W^T for power-of-two scales (the *_pow2 quantizers' output) on
    the block-scaled MMA; returns BF16 [m, n]."""
    _need(xq, torch.uint8, "xq")
    _need(wq, torch.uint8, "wq")
    m, k = xq.shape
    n = wq.shape[0]
    y = torch.empty((m, n), dtype=torch.bfloat16, device=xq.device) if y is None else y
    _check("fp8_block_gemm_pow2", lib().fp8_block_gemm_pow2(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws),
                                                            _ptr(y), m, n, k, _stream(stream)))
    return y


def fp8_grouped_gemm(xq, xs, row_idx, group_offsets, total_rows, wq, ws, y=None, stream=None):
    """Per-expert GEMM over routed rows.  wq [g, n, k], ws [g, ceil(n/128),
    ceil(k/128)], group_offsets int32 [g+1] (device), row_idx int32 [total]
    or None; total_rows is the host value of group_offsets[g]."""
    _need(xq, torch.uint8, "xq")
    _need(wq, torch.uint8, "wq")
    g, n, k = wq.shape
    y = torch.empty((total_rows, n), dtype=torch.bfloat16, device=xq.device) if y is None else y
    _check("fp8_grouped_gemm",
           lib().fp8_grouped_gemm(_ptr(xq), _ptr(xs), xq.shape[0], _ptr(row_idx), _ptr(group_offsets),
                                  g, int(total_rows), _ptr(wq), _ptr(ws), _ptr(y), n, k,
                                  _stream(stream)))
    return y


LINEAR_SINGLE_KERNEL = 2


def w8a8_linear(x, wq, ws, y=None, xq=None, xs=None, stream=None, static_weights=False,
                single_kernel=False, return_codes=False):
    """BF16 activations [m, k] -> 1x128 quantization -> blockwise FP8 GEMM
    (the C entry point w8a8_linear).  xq/xs, the activations' codes and
    scales, are written when given; they are allocated here unless the one
    kernel way runs (m <= 128 and k <= 32768, with n <= 1024 or
    single_kernel) and return_codes is off.  Returns y, or (y, xq, xs) with
    return_codes."""
    _need(x, torch.bfloat16, "x")
    _need(wq, torch.uint8, "wq")
    m, k = x.shape
    n = wq.shape[0]
    y = torch.empty((m, n), dtype=torch.bfloat16, device=x.device) if y is None else y
    one_kernel = m <= 128 and k <= 32768 and (single_kernel or n <= 1024)
    if xq is None and (return_codes or not one_kernel):
        xq = torch.empty((m, k), dtype=torch.uint8, device=x.device)
        xs = torch.empty((m, _cdiv(k, 128)), dtype=torch.float32, device=x.device)
    flags = (GEMM_STATIC_WEIGHTS if static_weights else 0) | (LINEAR_SINGLE_KERNEL if single_kernel else 0)
    _check("w8a8_linear", lib().w8a8_linear(_ptr(x), m, k, _ptr(wq), _ptr(ws), n, _ptr(y),
                                            _ptr(xq), _ptr(xs), flags, _stream(stream)))
    return (y, xq, xs) if return_codes else y


# --------------------------------------------------------------- KV cache

def kv_amax_quantize(x, q=None, scale=None, amax=None, mode=KV_AMAX_AND_QUANT, stream=None):
    """Per-tensor FP8 quantization with amax recalibration.  Returns
    (q uint8 like x, scale float32 [1], amax float32 [1])."""
    _need(x, torch.bfloat16, "x")
    dev = x.device
    if q is None and mode != KV_AMAX_ONLY:
        q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    scale = torch.empty(1, dtype=torch.float32, device=dev) if scale is None else scale
    if amax is None and mode != KV_QUANT_ONLY:
        amax = torch.empty(1, dtype=torch.float32, device=dev)
    _check("kv_amax_quantize", lib().kv_amax_quantize(_ptr(x), x.numel(), _ptr(q), _ptr(scale),
                                                      _ptr(amax), mode, _stream(stream)))
    return q, scale, amax


def consume_device_error():
    """Reads and clears the error code a GEMM kernel records when one of its
    bounded waits gives up (0 = none)."""
    v = ctypes.c_int(0)
    _check("w8a8_consume_device_error", lib().w8a8_consume_device_error(ctypes.byref(v)))
    return v.value


def debug_force_wait_timeout(on):
    """Test hook: while on, the GEMMs and the weight quantizer behave as if a
    bounded wait had run out of time (see w8a8_debug_force_wait_timeout)."""
    _check("w8a8_debug_force_wait_timeout", lib().w8a8_debug_force_wait_timeout(1 if on else 0))
