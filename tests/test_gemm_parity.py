"""GPU parity of the blockwise FP8 GEMM and its grouped (MoE) variant against
the CPU oracle's exact result, within the stated tolerance
(1e-3 * sum|a b| + half a BF16 ulp) and a tight one (2^-14 * sum|a b|)."""
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


def _scales(shape, seed, lo=1e-3, hi=3e-2):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(*shape, generator=g, dtype=torch.float64) * (hi - lo) + lo).float().numpy()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _cdiv(a, b):
    return -(-a // b)


GEMM_SHAPES = [(1, 16, 128), (3, 136, 256), (128, 256, 512), (200, 512, 384), (257, 264, 1024),
               (64, 256, 144), (130, 520, 256), (1, 8, 16), (256, 1024, 4096), (129, 768, 12288),
               # m <= 256 runs the weight-streaming kernel: token paddings 32/64/128/256,
               # K splits of 1..8 (one 128-row tile over 32 slabs splits 8 ways), ragged
               # N tiles and a partial last K slab
               (32, 128, 4096), (33, 256, 1024), (65, 384, 2048), (255, 136, 12288),
               (17, 1160, 400), (96, 128, 256),
               # 256 rows: the cluster reduction in one round (splits up to 4) or in
               # rounds of 128 rows
               (256, 4096, 1024), (250, 2048, 2048),
               # few rows but K past the weight-streaming kernel's reach: the general kernel
               (3, 128, 32896)]


@pytest.mark.parametrize("m,n,k", GEMM_SHAPES)
def test_block_gemm_small(W, m, n, k):
    xq, wq = _codes((m, k), m + k), _codes((n, k), n + 7 * k)
    xs, ws = _scales((m, _cdiv(k, 128)), 1), _scales((_cdiv(n, 128), _cdiv(k, 128)), 2)
    y = W.fp8_block_gemm(_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    y_ref, absref = O.block_gemm(xq, xs, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, f"gemm {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [sh for sh in GEMM_SHAPES if sh[0] <= 256])
def test_block_gemm_static_weights_same_bits(W, m, n, k):
    """The static-weights flag changes when the weights are read, not what
    is computed: the same bits as without it."""
    xq, wq = _codes((m, k), m + k), _codes((n, k), n + 7 * k)
    xs, ws = _scales((m, _cdiv(k, 128)), 1), _scales((_cdiv(n, 128), _cdiv(k, 128)), 2)
    args = (_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    y0 = W.fp8_block_gemm(*args)
    y1 = W.fp8_block_gemm(*args, static_weights=True)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


@pytest.mark.parametrize("m", [1, 64, 200])
def test_decode_chain_static_weights(W, m):
    """A chain of dependent linears on one stream, as in a decode step:
    each GEMM's BF16 output is quantized (1x128) and feeds the next GEMM.
    With static weights each GEMM may start streaming its weights while the
    previous kernel runs, but must read its activations only after it: the
    chain's result is bit-identical to the one without the flag."""
    dims = [1024, 2048, 1024, 3072, 1024, 1024]
    ws_ = [W.quantize_weight_blockwise(synth.weights(dims[i + 1], dims[i], seed=70 + i).cuda())
           for i in range(len(dims) - 1)]
    x0 = synth.activations(m, dims[0], seed=69).cuda()

    def chain(static):
        x = x0
        for wq, wsc in ws_:
            xq, xs = W.quantize_act_per_token_group(x)
            x = W.fp8_block_gemm(xq, xs, wq, wsc, static_weights=static)
        return x

    ya = chain(False)
    yb = chain(True)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))


@pytest.mark.parametrize("m,n,k", [(2305, 2312, 48), (5000, 776, 32), (1100, 2312, 48)])
def test_block_gemm_partial_last_n_tile_several_waves(W, m, n, k):
    """More tiles than SMs, with a last N tile of 8 columns: a CTA's epilogue
    stores that tile with a single TMA store and starts its next tile at once.
    Called three times, since a staging-buffer race shows only in some runs.
    1100 x 2312 runs the 128-wide tiles (90 tiles 256 wide, 171 128 wide)."""
    xq, wq = _codes((m, k), m + k), _codes((n, k), n + 7 * k)
    xs, ws = _scales((m, _cdiv(k, 128)), 1), _scales((_cdiv(n, 128), _cdiv(k, 128)), 2)
    y_ref, absref = O.block_gemm(xq, xs, wq, ws)
    args = (_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    for rep in range(3):
        y = W.fp8_block_gemm(*args)
        torch.cuda.synchronize()
        assert W.consume_device_error() == 0
        assert_gemm_close(bits16(y), y_ref, absref, f"gemm {m}x{n}x{k} call {rep}")


def test_block_gemm_empty_and_k0(W):
    y = W.fp8_block_gemm(torch.empty(0, 128, dtype=torch.uint8, device="cuda"),
                         torch.empty(0, 1, device="cuda"),
                         torch.zeros(256, 128, dtype=torch.uint8, device="cuda"),
                         torch.ones(2, 1, device="cuda"))
    assert y.shape == (0, 256)
    y = torch.full((5, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    W.fp8_block_gemm(torch.empty(5, 0, dtype=torch.uint8, device="cuda"),
                     torch.empty(5, 0, device="cuda"),
                     torch.empty(256, 0, dtype=torch.uint8, device="cuda"),
                     torch.empty(2, 0, device="cuda"), y=y)
    torch.cuda.synchronize()
    assert (y == 0).all()


def test_single_w8a8_linear_config(W):
    """X [128, 512] ~ N(0,1) with 0.1% x50 outliers, W [256, 512] ~ N(0, 0.02),
    seed 0: quantized by the oracle, multiplied on the GPU."""
    x = synth.activations(128, 512, seed=0)
    w = synth.weights(256, 512, seed=1)
    xq, xs = O.quantize_act_per_token_group(synth.bf16_bits(x))
    wq, ws = O.quantize_weight_blockwise(synth.bf16_bits(w))
    y = W.fp8_block_gemm(_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    torch.cuda.synchronize()
    y_ref, absref = O.block_gemm(xq, xs, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, "config-1 linear")
    # and through the linear from BF16 (quantization fused into the GEMM)
    y2 = W.w8a8_linear(x.cuda(), _dev(wq), _dev(ws))
    torch.cuda.synchronize()
    assert_gemm_close(bits16(y2), y_ref, absref, "config-1 linear, fused")


def test_linear_with_power_of_two_scales(W):
    """The GEMM takes power-of-two scales as they come: both operands
    quantized on the GPU with pow2 scales (bit-exact with the oracle's), then
    the GEMM within the tolerance of the oracle's exact product."""
    x = synth.activations(200, 1024, seed=8)
    w = synth.weights(384, 1024, seed=9)
    xq, xs = W.quantize_act_per_token_group(x.cuda(), pow2=True)
    wq, ws = W.quantize_weight_blockwise(w.cuda(), pow2=True)
    y = W.fp8_block_gemm(xq, xs, wq, ws)
    torch.cuda.synchronize()
    xq_r, xs_r = O.quantize_blocks(synth.bf16_bits(x), 1, 128, pow2=True)
    wq_r, ws_r = O.quantize_blocks(synth.bf16_bits(w), 128, 128, pow2=True)
    assert (xq.cpu().numpy() == xq_r).all() and (wq.cpu().numpy() == wq_r).all()
    y_ref, absref = O.block_gemm(xq_r, xs_r, wq_r, ws_r)
    assert_gemm_close(bits16(y), y_ref, absref, "pow2 linear")


def test_scale_power_of_two_is_exact(W):
    m, n, k = 96, 512, 1024
    xq, wq = _codes((m, k), 3), _codes((n, k), 4)
    xs, ws = _scales((m, 8), 5), _scales((4, 8), 6)
    y1 = W.fp8_block_gemm(_dev(xq), _dev(xs), _dev(wq), _dev(ws))
    y2 = W.fp8_block_gemm(_dev(xq), _dev(xs), _dev(wq), _dev(ws * np.float32(4)))
    torch.cuda.synchronize()
    assert torch.equal(y1.float() * 4, y2.float())


@pytest.mark.parametrize("m", [1, 64, 128, 256, 8192])
def test_block_gemm_qwen3_8b_shapes_sampled(W, m):
    """The four Qwen3-8B linears at M tokens, full size, checked on sampled
    entries: every tile corner of a tile row plus random positions."""
    rng = np.random.default_rng(m)
    for j, (name, (n, k)) in enumerate(synth.QWEN3_8B_LINEARS.items()):
        xq, wq = _codes((m, k), 10 * m + j), _codes((n, k), 20 * m + j, spread=100)
        xs, ws = _scales((m, k // 128), 30 + j), _scales((n // 128, k // 128), 40 + j, 1e-4, 1e-3)
        y = W.fp8_block_gemm(_dev(xq), _dev(xs), _dev(wq), _dev(ws))
        torch.cuda.synchronize()
        assert W.consume_device_error() == 0
        ii = np.concatenate([rng.integers(0, m, 3000), np.repeat([0, m - 1, min(m - 1, 127), min(m - 1, 128)], 64)])
        jj = np.concatenate([rng.integers(0, n, 3000), np.tile(np.linspace(0, n - 1, 64).astype(np.int64), 4)])
        y_ref, absref = O.block_gemm_entries(xq, xs, wq, ws, ii, jj)
        assert_gemm_close(bits16(y)[ii, jj], y_ref, absref, f"{name} m={m}")


# ------------------------------------------------------------- grouped

def _grouped_case(g, n, k, rows_x, total, seed, gather=True, bad_rows=False):
    rng = np.random.default_rng(seed)
    xq = _codes((rows_x, k), seed)
    xs = _scales((rows_x, _cdiv(k, 128)), seed + 1)
    wq = _codes((g, n, k), seed + 2)
    ws = _scales((g, _cdiv(n, 128), _cdiv(k, 128)), seed + 3)
    cuts = np.sort(rng.integers(0, total + 1, g - 1))
    off = np.concatenate([[0], cuts, [total]]).astype(np.int32)
    row_idx = rng.integers(0, rows_x, total).astype(np.int32) if gather else None
    if bad_rows and gather:
        row_idx[::17] = -1
        row_idx[5::23] = rows_x
    return xq, xs, wq, ws, off, row_idx


def test_grouped_gemm_partial_last_n_tile_several_waves(W):
    """Grouped tiles outnumbering the SMs, each expert's last N tile 8 columns
    wide; three calls (the staging-buffer race showed only in some runs)."""
    g, n, k, rows_x, total = 4, 520, 32, 3000, 8000
    xq, xs, wq, ws, off, row_idx = _grouped_case(g, n, k, rows_x, total, seed=77)
    y_ref, absref = O.grouped_gemm(xq, xs, row_idx, off, wq, ws)
    args = (_dev(xq), _dev(xs), _dev(row_idx), _dev(off), total, _dev(wq), _dev(ws))
    for rep in range(3):
        y = W.fp8_grouped_gemm(*args)
        torch.cuda.synchronize()
        assert W.consume_device_error() == 0
        assert_gemm_close(bits16(y), y_ref, absref, f"grouped partial-N call {rep}")


@pytest.mark.parametrize("g,n,k,rows_x,total,gather", [
    (5, 264, 256, 40, 300, True), (3, 256, 128, 500, 500, False), (1, 512, 384, 300, 300, False),
    (8, 128, 768, 64, 700, True), (4, 1536, 2048, 100, 260, True), (2, 2048, 768, 300, 300, False)])
def test_grouped_gemm_small(W, g, n, k, rows_x, total, gather):
    xq, xs, wq, ws, off, row_idx = _grouped_case(g, n, k, rows_x, total, seed=g * 100 + n, gather=gather)
    y = W.fp8_grouped_gemm(_dev(xq), _dev(xs), None if row_idx is None else _dev(row_idx), _dev(off),
                           total, _dev(wq), _dev(ws))
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    y_ref, absref = O.grouped_gemm(xq, xs, row_idx, off, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, f"grouped g={g} n={n} k={k}")


def test_grouped_gemm_out_of_range_rows_give_zero(W):
    xq, xs, wq, ws, off, row_idx = _grouped_case(3, 256, 256, 50, 200, seed=9, gather=True, bad_rows=True)
    y = W.fp8_grouped_gemm(_dev(xq), _dev(xs), _dev(row_idx), _dev(off), 200, _dev(wq), _dev(ws))
    torch.cuda.synchronize()
    yb = bits16(y)
    bad = (row_idx < 0) | (row_idx >= 50)
    assert (yb[bad] == 0).all()
    ok = ~bad
    safe = np.where(ok, row_idx, 0).astype(np.int32)
    y_ref, absref = O.grouped_gemm(xq, xs, safe, off, wq, ws)
    assert_gemm_close(yb[ok], y_ref[ok], absref[ok], "grouped with bad rows")


def test_grouped_single_group_identity_equals_dense(W):
    m, n, k = 300, 512, 1024
    xq, wq = _codes((m, k), 1), _codes((1, n, k), 2)
    xs, ws = _scales((m, 8), 3), _scales((1, 4, 8), 4)
    yd = W.fp8_block_gemm(_dev(xq), _dev(xs), _dev(wq[0]), _dev(ws[0]))
    yg = W.fp8_grouped_gemm(_dev(xq), _dev(xs), None, _dev(np.array([0, m], np.int32)), m, _dev(wq), _dev(ws))
    torch.cuda.synchronize()
    assert torch.equal(yd, yg)


def test_moe_layer_qwen3_30b_a3b_sampled(W):
    """One Qwen3-30B-A3B MoE layer: 4096 tokens routed top-8 over 128 experts;
    gate_up [1536, 2048] over gathered token rows, down [2048, 768] over the
    routed rows.  Full size, checked on sampled routed rows and columns."""
    T, H, E, I, K8 = synth.MOE_TOKENS, synth.MOE_HIDDEN, synth.MOE_EXPERTS, synth.MOE_INTER, synth.MOE_TOPK
    r = synth.moe_routing(T, E, K8, seed=4)
    total = T * K8
    off = r.group_offsets.numpy()
    row_idx = r.row_idx.numpy()
    rng = np.random.default_rng(4)
    cases = [("gate_up", 2 * I, H, T, row_idx), ("down", H, I, total, None)]
    for name, n, k, rows_x, ri in cases:
        xq = _codes((rows_x, k), n)
        xs = _scales((rows_x, k // 128), n + 1)
        wq = _codes((E, n, k), n + 2, spread=100)
        ws = _scales((E, n // 128, k // 128), n + 3, 1e-4, 1e-3)
        y = W.fp8_grouped_gemm(_dev(xq), _dev(xs), None if ri is None else _dev(ri), _dev(off), total,
                               _dev(wq), _dev(ws))
        torch.cuda.synchronize()
        assert W.consume_device_error() == 0
        yb = bits16(y)
        rows = np.concatenate([off[:-1][np.diff(off) > 0], off[1:][np.diff(off) > 0] - 1,
                               rng.integers(0, total, 200)])
        cols = rng.integers(0, n, 64)
        for rr in rows:
            e = int(np.searchsorted(off, rr, side="right") - 1)
            src = rr if ri is None else ri[rr]
            y_ref, absref = O.block_gemm_entries(xq[src:src + 1], xs[src:src + 1], wq[e], ws[e],
                                                 np.zeros_like(cols), cols)
            assert_gemm_close(yb[rr, cols], y_ref, absref, f"moe {name} row {rr}")
