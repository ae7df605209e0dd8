"""GPU parity of the power-of-two-scale GEMM (the block-scaled MMA path)
against the CPU oracle's exact result, within the stated tolerance
(1e-3 * sum|a b| + half a BF16 ulp) and the tight one (2^-14 * sum|a b|)."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import assert_gemm_close, bits16
from w8a8_gemm_rl_gb300 import synth

pytestmark = pytest.mark.gpu


def _codes(shape, seed, spread=60.0):
    """E4M3 codes of N(0, spread) values (library conversion, in range)."""
    g = torch.Generator().manual_seed(seed)
    v = (torch.randn(*shape, generator=g) * spread).clamp_(-448, 448)
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _pow2_scales(shape, seed, lo=-12, hi=-4):
    """2^e with e uniform in [lo, hi]."""
    rng = np.random.default_rng(seed)
    return np.ldexp(np.float32(1), rng.integers(lo, hi + 1, shape)).astype(np.float32)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _cdiv(a, b):
    return -(-a // b)


# sized so that the oracle's exact product takes seconds
SHAPES = [(1, 16, 128), (3, 136, 256), (128, 256, 512), (200, 512, 384), (257, 264, 1024),
          (64, 256, 144), (130, 520, 256), (1, 8, 16), (256, 512, 4096), (129, 768, 2048),
          # nine M tiles (a partial raster group) with ragged M, N and K tails
          (1100, 520, 272),
          # 257 K slabs: the operand and scale rings wrap many times
          (3, 264, 32896)]


@pytest.mark.parametrize("m,n,k", SHAPES)
def test_pow2_gemm_small(W, m, n, k):
    xq, wq = _codes((m, k), m + k), _codes((n, k), n + 7 * k)
    xs = _pow2_scales((m, _cdiv(k, 128)), 1)
    ws = _pow2_scales((_cdiv(n, 128), _cdiv(k, 128)), 2)
    y = W.fp8_block_gemm_pow2(_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    y_ref, absref = O.block_gemm(xq, xs, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, f"pow2 gemm {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [(2305, 2312, 48), (5000, 776, 32)])
def test_pow2_gemm_partial_last_n_tile_several_waves(W, m, n, k):
    """More tiles than SMs, with a last N tile of 8 columns, called three
    times: a staging-buffer race once corrupted that tile in some runs."""
    xq, wq = _codes((m, k), m + k), _codes((n, k), n + 7 * k)
    xs = _pow2_scales((m, _cdiv(k, 128)), 1)
    ws = _pow2_scales((_cdiv(n, 128), _cdiv(k, 128)), 2)
    y_ref, absref = O.block_gemm(xq, xs, wq, ws)
    args = (_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    for rep in range(3):
        y = W.fp8_block_gemm_pow2(*args)
        torch.cuda.synchronize()
        assert W.consume_device_error() == 0
        assert_gemm_close(bits16(y), y_ref, absref, f"pow2 gemm {m}x{n}x{k} call {rep}")


@pytest.mark.parametrize("xe,we", [((-127, -126, -120), (100, 120, 127)),
                                   ((100, 120, 127), (-127, -126, -120))])
def test_pow2_gemm_extreme_exponents(W, xe, we):
    """Scales at both ends of the UE8M0 range (2^-127, a binary32 subnormal,
    and 2^127), paired so that every scaled product stays finite."""
    m, n, k = 256, 512, 512
    xq, wq = _codes((m, k), 11), _codes((n, k), 12)
    rng = np.random.default_rng(13)
    xs = np.ldexp(np.float32(1), rng.choice(xe, size=(m, 4))).astype(np.float32)
    ws = np.ldexp(np.float32(1), rng.choice(we, size=(4, 4))).astype(np.float32)
    y = W.fp8_block_gemm_pow2(_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    y_ref, absref = O.block_gemm(xq, xs, wq, ws)
    assert np.isfinite(y_ref).all() and (absref < 2.0 ** 100).all()
    assert_gemm_close(bits16(y), y_ref, absref, f"pow2 exponents {xe} x {we}")


def test_pow2_linear_from_quantizers(W):
    """Both operands quantized on the GPU with power-of-two scales (bit-exact
    with the oracle's), then this GEMM within the tolerance of the oracle's
    exact product of the oracle's codes."""
    x = synth.activations(200, 1024, seed=8)
    w = synth.weights(384, 1024, seed=9)
    xq, xs = W.quantize_act_per_token_group(x.cuda(), pow2=True)
    wq, ws = W.quantize_weight_blockwise(w.cuda(), pow2=True)
    y = W.fp8_block_gemm_pow2(xq, xs, wq, ws)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    xq_r, xs_r = O.quantize_blocks(synth.bf16_bits(x), 1, 128, pow2=True)
    wq_r, ws_r = O.quantize_blocks(synth.bf16_bits(w), 128, 128, pow2=True)
    assert (xq.cpu().numpy() == xq_r).all() and (wq.cpu().numpy() == wq_r).all()
    assert (xs.cpu().numpy() == xs_r).all() and (ws.cpu().numpy() == ws_r).all()
    y_ref, absref = O.block_gemm(xq_r, xs_r, wq_r, ws_r)
    assert_gemm_close(bits16(y), y_ref, absref, "pow2 linear")


def test_pow2_scaling_is_exact(W):
    """Doubling every weight scale doubles every output exactly."""
    m, n, k = 300, 512, 1024
    xq, wq = _codes((m, k), 3), _codes((n, k), 4)
    xs, ws = _pow2_scales((m, 8), 5), _pow2_scales((4, 8), 6)
    y1 = W.fp8_block_gemm_pow2(_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    y2 = W.fp8_block_gemm_pow2(_dev(xq), _dev(xs), _dev(wq), _dev(ws * np.float32(2)))
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    assert torch.equal(y1.float() * 2, y2.float())


@pytest.mark.parametrize("m", [257, 8192])
def test_pow2_gemm_qwen3_8b_shapes_sampled(W, m):
    """The four Qwen3-8B linears at M tokens, full size, checked on sampled
    entries: tile corners of the first and last tile rows plus random
    positions."""
    rng = np.random.default_rng(m)
    for j, (name, (n, k)) in enumerate(synth.QWEN3_8B_LINEARS.items()):
        xq, wq = _codes((m, k), 10 * m + j), _codes((n, k), 20 * m + j, spread=100)
        xs = _pow2_scales((m, k // 128), 30 + j)
        ws = _pow2_scales((n // 128, k // 128), 40 + j, -14, -10)
        y = W.fp8_block_gemm_pow2(_dev(xq), _dev(xs), _dev(wq), _dev(ws))
        torch.cuda.synchronize()
        assert W.consume_device_error() == 0
        ii = np.concatenate([rng.integers(0, m, 3000), np.repeat([0, m - 1, 127, 128], 64)])
        jj = np.concatenate([rng.integers(0, n, 3000), np.tile(np.linspace(0, n - 1, 64).astype(np.int64), 4)])
        y_ref, absref = O.block_gemm_entries(xq, xs, wq, ws, ii, jj)
        assert_gemm_close(bits16(y)[ii, jj], y_ref, absref, f"pow2 {name} m={m}")


def test_pow2_gemm_rejects_scales_it_cannot_hold(W):
    """A scale that is not a power of two, or below 2^-127, is reported as
    device error 59; the call completes and the next good call is exact."""
    m, n, k = 200, 256, 512
    xq, wq = _codes((m, k), 21), _codes((n, k), 22)
    xs, ws = _pow2_scales((m, 4), 23), _pow2_scales((2, 4), 24)
    assert W.consume_device_error() == 0
    for bad in (np.float32(3.0), np.float32(2.0 ** -130)):
        ws_bad = ws.copy()
        ws_bad[1, 2] = bad
        W.fp8_block_gemm_pow2(_dev(xq), _dev(xs), _dev(wq), _dev(ws_bad))
        torch.cuda.synchronize()
        assert W.consume_device_error() == 59
    y = W.fp8_block_gemm_pow2(_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    y_ref, absref = O.block_gemm(xq, xs, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, "pow2 after bad scales")


def test_pow2_gemm_empty_and_k0(W):
    y = W.fp8_block_gemm_pow2(torch.empty(0, 128, dtype=torch.uint8, device="cuda"),
                              torch.empty(0, 1, device="cuda"),
                              torch.zeros(256, 128, dtype=torch.uint8, device="cuda"),
                              torch.ones(2, 1, device="cuda"))
    assert y.shape == (0, 256)
    y = torch.full((5, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    W.fp8_block_gemm_pow2(torch.empty(5, 0, dtype=torch.uint8, device="cuda"),
                          torch.empty(5, 0, device="cuda"),
                          torch.empty(256, 0, dtype=torch.uint8, device="cuda"),
                          torch.empty(2, 0, device="cuda"), y=y)
    torch.cuda.synchronize()
    assert (y == 0).all()
