"""GPU parity of the dequantizer (fake quant) and the quantization-error
report against the CPU oracle: BF16 outputs bit for bit; report maxima
exactly and sums within the documented 1e-5 relative."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import bits16, u8
from w8a8_gemm_rl_gb300 import synth

pytestmark = pytest.mark.gpu

DEQUANT_CASES = [  # rows, cols, block_rows, block_cols
    (256, 512, 128, 128), (300, 200, 128, 128), (64, 768, 1, 128), (7, 1000, 1, 128),
    (1, 4096, 1, 4096), (5, 24, 1, 128), (3, 7, 2, 3), (0, 128, 1, 128), (129, 144, 128, 128)]


def _codes_and_scales(rows, cols, br, bc, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.int32)
    q[(q & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    q = q.to(torch.uint8)
    s = torch.exp(torch.randn((-(-rows // br), -(-cols // bc)), generator=g) * 4.0).float()
    return q, s


@pytest.mark.parametrize("rows,cols,br,bc", DEQUANT_CASES)
def test_dequantize_bit_exact(W, rows, cols, br, bc):
    q, s = _codes_and_scales(rows, cols, br, bc, seed=rows * 131 + cols)
    y = W.dequantize_blockwise(q.cuda(), s.cuda(), br, bc)
    want = O.dequantize_blocks(q.numpy(), s.numpy(), br, bc)
    assert (bits16(y) == want).all()


def test_dequantize_of_quantized_weights_and_kv(W):
    w = synth.weights(384, 640, seed=3, device="cuda")
    wq, ws = W.quantize_weight_blockwise(w)
    y = W.dequantize_blockwise(wq, ws, 128, 128)
    assert (bits16(y) == O.dequantize_blocks(u8(wq), ws.cpu().numpy(), 128, 128)).all()
    kv = synth.kv_cache(seed=4, shape=(2, 64, 8, 128), device="cuda")
    kq, ks, _ = W.kv_amax_quantize(kv)
    n = kv.numel()
    y = W.dequantize_blockwise(kq.reshape(1, n), ks.reshape(1, 1), 1, n)
    want = O.dequantize_blocks(u8(kq).reshape(1, n), ks.cpu().numpy().reshape(1, 1), 1, n)
    assert (bits16(y) == want).all()


REPORT_CASES = [  # rows, cols, quant block, report block
    (256, 512, (128, 128), (128, 128)), (64, 768, (1, 128), (1, 128)),
    (300, 200, (128, 128), (64, 64)), (1, 65536, (1, 65536), (1, 4096)),
    (7, 100, (1, 128), (7, 100)), (33, 4096, (1, 128), (33, 128)), (50, 100, (1, 128), (50, 100))]


@pytest.mark.parametrize("rows,cols,qb,rb", REPORT_CASES)
def test_quant_error_report_matches_oracle(W, rows, cols, qb, rb):
    x = synth.activations(rows, cols, seed=rows + cols, device="cuda")
    xb = synth.bf16_bits(x)
    q_ref, s_ref = O.quantize_blocks(xb, *qb)
    q = torch.from_numpy(q_ref).cuda()
    s = torch.from_numpy(s_ref).cuda()
    st = W.quant_error_report(x, q, s, qb, rb).cpu().numpy()
    want = O.quant_error(xb, q_ref, s_ref, qb[0], qb[1], rb[0], rb[1])
    assert st.shape == want.shape
    assert (st[..., 0] == want[..., 0]).all()
    assert np.allclose(st[..., 1:], want[..., 1:], rtol=1e-5, atol=0)
    # SQNR of E4M3 with block scales on N(0,1) data with outliers: 10-45 dB
    assert 10.0 < W.sqnr_db(torch.from_numpy(st)) < 45.0


def test_weight_sync_rows_at_full_size(W):
    """One Qwen3-8B gate_up matrix [24576, 4096] (the largest of the weight
    sync): power-of-two block quantization, dequantization and the error
    report, each checked against the oracle on sampled 128 x 128 blocks
    (blocks are independent, so a block alone gives the same result); the
    last block row and column included."""
    n, k = 24576, 4096
    w = synth.weights(n, k, seed=17, device="cuda")
    wq, ws = W.quantize_weight_blockwise(w, pow2=True)
    y = W.dequantize_blockwise(wq, ws, 128, 128)
    st = W.quant_error_report(w, wq, ws, (128, 128), (128, 128))
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(5)
    picks = [(0, 0), (n // 128 - 1, k // 128 - 1)] + [
        (int(torch.randint(0, n // 128, (1,), generator=g)), int(torch.randint(0, k // 128, (1,), generator=g)))
        for _ in range(6)]
    for bi, bj in picks:
        r, c = slice(128 * bi, 128 * bi + 128), slice(128 * bj, 128 * bj + 128)
        xb = synth.bf16_bits(w[r, c])
        q_ref, s_ref = O.quantize_blocks(xb, 128, 128, pow2=True)
        assert (u8(wq[r, c]) == q_ref).all()
        assert ws[bi, bj].item() == s_ref[0, 0]
        assert (bits16(y[r, c]) == O.dequantize_blocks(q_ref, s_ref, 128, 128)).all()
        want = O.quant_error(xb, q_ref, s_ref, 128, 128, 128, 128)[0, 0]
        got = st[bi, bj].cpu().numpy()
        assert got[0] == want[0]
        assert np.allclose(got[1:], want[1:], rtol=1e-5, atol=0)


BATCH_SHAPES = [(256, 512), (300, 208), (129, 1024), (8, 128), (0, 256), (384, 4096), (131, 16)]


def test_batched_dequantize_and_report(W):
    """Many matrices in one call each (128 x 128 blocks), ragged edges
    included: the dequantized BF16 bit-exact with the oracle, the report's
    maxima exact and sums within 1e-5, per matrix."""
    xs, qs, ss = [], [], []
    for i, (n, k) in enumerate(BATCH_SHAPES):
        x = synth.activations(n, k, seed=40 + i) if n else torch.zeros((0, k), dtype=torch.bfloat16)
        q_ref, s_ref = O.quantize_blocks(synth.bf16_bits(x), 128, 128)
        xs.append(x.cuda())
        qs.append(torch.from_numpy(q_ref).cuda())
        ss.append(torch.from_numpy(s_ref).cuda())
    ys = W.dequantize_blockwise_batched(qs, ss)
    sts = W.quant_error_report_batched(xs, qs, ss)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    for x, q, s, y, st in zip(xs, qs, ss, ys, sts):
        if x.shape[0] == 0:
            continue
        q_ref, s_ref = q.cpu().numpy(), s.cpu().numpy()
        assert (bits16(y) == O.dequantize_blocks(q_ref, s_ref, 128, 128)).all()
        want = O.quant_error(synth.bf16_bits(x.cpu()), q_ref, s_ref, 128, 128, 128, 128)
        got = st.cpu().numpy()
        assert (got[..., 0] == want[..., 0]).all()
        assert np.allclose(got[..., 1:], want[..., 1:], rtol=1e-5, atol=0)


def test_batched_equals_one_matrix_calls(W):
    """The batched dequantizer gives the one-matrix call's bits on a weight
    sync's matrices (one Qwen3-8B layer)."""
    ws_ = [W.quantize_weight_blockwise(synth.weights(n, k, seed=50 + i, device="cuda"))
           for i, (n, k) in enumerate(synth.QWEN3_8B_LINEARS.values())]
    ys = W.dequantize_blockwise_batched([q for q, _ in ws_], [s for _, s in ws_])
    for (q, s), y in zip(ws_, ys):
        assert torch.equal(y.view(torch.int16), W.dequantize_blockwise(q, s, 128, 128).view(torch.int16))
