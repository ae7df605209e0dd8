"""GPU parity of w8a8_linear, the W8A8 linear from BF16 activations: for
m <= 128 a single kernel whose token loaders quantize each 1 x 128 group on
the way into shared memory.  The codes and scales it writes out are checked
bit for bit against the oracle's activation quantizer, and Y against the
oracle's exact product of those codes (1e-3 contract and the 2^-14 tight
bound)."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import assert_gemm_close, bits16
from w8a8_gemm_rl_gb300 import synth

pytestmark = pytest.mark.gpu

LINEAR_SHAPES = [(1, 256, 512), (37, 384, 1024), (64, 1024, 4096), (128, 264, 12288),
                 (100, 512, 400), (33, 128, 4096), (128, 6144, 256), (5, 4096, 32768)]


def _case(m, n, k, seed):
    x = synth.activations(m, k, seed=seed)
    if m > 3:
        x[1] = 0.0                       # an all-zero row: S = 1, codes 0
        x[2] = -0.0                      # signed zeros keep their sign: codes 0x80
    w = synth.weights(n, k, seed=seed + 1)
    wq, ws = O.quantize_weight_blockwise(synth.bf16_bits(w))
    return x, wq, ws


@pytest.mark.parametrize("single", [False, True])
@pytest.mark.parametrize("m,n,k", LINEAR_SHAPES)
def test_linear_codes_exact_and_y_within_tolerance(W, m, n, k, single):
    """Either way of running it (one fused kernel, or quantizer + GEMM)."""
    x, wq, ws = _case(m, n, k, seed=m + n + k)
    y, xq, xs = W.w8a8_linear(x.cuda(), torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda(),
                              single_kernel=single, return_codes=True)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    xq_ref, xs_ref = O.quantize_act_per_token_group(synth.bf16_bits(x))
    assert (xq.cpu().numpy() == xq_ref).all()
    assert (xs.cpu().numpy() == xs_ref).all()
    y_ref, absref = O.block_gemm(xq_ref, xs_ref, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, f"linear {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [(64, 1024, 4096), (100, 512, 400), (64, 6144, 4096)])
def test_linear_without_code_outputs(W, m, n, k):
    """Without xq/xs (NULL) the one-kernel way writes only y: the same bits."""
    x, wq, ws = _case(m, n, k, seed=7)
    args = (x.cuda(), torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda())
    y1, _, _ = W.w8a8_linear(*args, single_kernel=True, return_codes=True)
    y2 = W.w8a8_linear(*args, single_kernel=True)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_linear_two_kernel_path(W):
    """m > 128: the activation quantizer and the GEMM as two kernels."""
    m, n, k = 300, 512, 1024
    x, wq, ws = _case(m, n, k, seed=11)
    y, xq, xs = W.w8a8_linear(x.cuda(), torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda(),
                              return_codes=True)
    torch.cuda.synchronize()
    xq_ref, xs_ref = O.quantize_act_per_token_group(synth.bf16_bits(x))
    assert (xq.cpu().numpy() == xq_ref).all() and (xs.cpu().numpy() == xs_ref).all()
    y_ref, absref = O.block_gemm(xq_ref, xs_ref, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, "two-kernel linear")


@pytest.mark.parametrize("m", [1, 64, 128])
def test_fused_decode_chain_static_weights(W, m):
    """A chain of dependent fused linears (each output is the next input),
    as in a decode step; with static weights each may start streaming its
    weights while the previous kernel runs, but reads its activations only
    after it: the chain's output is bit-identical to the one without."""
    dims = [1024, 2048, 1024, 3072, 1024, 1024]
    ws_ = [W.quantize_weight_blockwise(synth.weights(dims[i + 1], dims[i], seed=90 + i).cuda())
           for i in range(len(dims) - 1)]
    x0 = synth.activations(m, dims[0], seed=89).cuda()

    def chain(static):
        x = x0
        for i, (wq, wsc) in enumerate(ws_):
            # alternate the two ways: quantizer + GEMM and one fused kernel
            x = W.w8a8_linear(x, wq, wsc, static_weights=static, single_kernel=bool(i % 2))
        return x

    ya = chain(False)
    yb = chain(True)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
    # and the last link against the oracle, from the GPU's own input to it
    x = x0
    for i, (wq, wsc) in enumerate(ws_[:-1]):
        x = W.w8a8_linear(x, wq, wsc, single_kernel=bool(i % 2))
    xq_ref, xs_ref = O.quantize_act_per_token_group(synth.bf16_bits(x.cpu()))
    wq, wsc = ws_[-1]
    y_ref, absref = O.block_gemm(xq_ref, xs_ref, wq.cpu().numpy(), wsc.cpu().numpy())
    assert_gemm_close(bits16(yb), y_ref, absref, f"chain m={m}")
