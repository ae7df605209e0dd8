"""GPU parity of the E4M3 codec and the three quantizers against the CPU
oracle: codes and scales must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle as O
from parity_util import bits16, f32, u8
from w8a8_gemm_rl_gb300 import synth

pytestmark = pytest.mark.gpu


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


# ------------------------------------------------------------------ codec

def test_e4m3_encode_every_binary32_pattern(W):
    """The hardware conversion behind every quantizer, against the oracle's
    encoder, on all 2^32 binary32 bit patterns (NaN inputs excluded)."""
    chunk = 1 << 27
    for start in range(0, 1 << 32, chunk):
        x = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda").to(torch.int32)
        q = W.e4m3_encode_f32(x.view(torch.float32))
        got = u8(q)
        want = O.e4m3_encode_patterns(start, chunk)
        pats = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32)
        nan = (pats & 0x7FFFFFFF) > 0x7F800000
        bad = (got != want) & ~nan
        assert not bad.any(), (hex(int(pats[bad][0])), hex(got[bad][0]), hex(want[bad][0]))


def test_e4m3_decode_all_codes(W):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).cuda()
    # pad to exercise the vector path (16 codes per thread) and the tail
    q = torch.cat([codes, codes, codes[:37]])
    x = f32(W.e4m3_decode_f32(q)).astype(np.float64)
    want = O.e4m3_decode(u8(q))
    nan = np.isnan(want)
    assert (np.isnan(x) == nan).all()
    assert (x[~nan] == want[~nan]).all()
    assert (np.signbit(x[~nan]) == np.signbit(want[~nan])).all()


# --------------------------------------------------------- act quantizer

GATHER_CASES = [  # rows_x, k, total routed rows
    (300, 2048, 1000), (50, 768, 400), (37, 200, 123), (64, 1024, 64), (10, 8, 33),
    (0, 256, 17), (5, 128, 0), (4096, 2048, 32768)]


@pytest.mark.parametrize("rows_x,k,total", GATHER_CASES)
def test_act_quant_gather_bit_exact(W, rows_x, k, total):
    """Routed-row quantizer: every row and scale equals the oracle's, including
    duplicated rows and indices outside [0, rows_x) (zero rows)."""
    x = synth.activations(max(rows_x, 1), k, seed=rows_x * 31 + k, device="cpu")[:rows_x]
    g = torch.Generator().manual_seed(rows_x + 7 * total)
    idx = torch.randint(-3, rows_x + 3, (total,), generator=g, dtype=torch.int64)
    if total >= 4:
        idx[:4] = torch.tensor([-(2 ** 31), 2 ** 31 - 1, 0, max(rows_x - 1, 0)])
    idx = idx.to(torch.int32)
    xq, xs = W.quantize_act_per_token_group_gather(x.cuda(), idx.cuda())
    q_ref, s_ref = O.quantize_act_per_token_group_gather(synth.bf16_bits(x), idx.numpy())
    assert (u8(xq) == q_ref).all()
    assert (f32(xs).view(np.uint32) == s_ref.view(np.uint32)).all()


def test_act_quant_gather_of_moe_routing_equals_quant_then_gather(W):
    """On the Qwen3-30B-A3B routing: quantizing the routed rows directly gives
    the gathered rows of the plain per-token quantization."""
    r = synth.moe_routing(4096, 128, 8, seed=60)
    x = synth.activations(4096, 2048, seed=61, device="cuda")
    xq, xs = W.quantize_act_per_token_group(x)
    gq, gs = W.quantize_act_per_token_group_gather(x, r.row_idx.cuda())
    ri = r.row_idx.cuda().long()
    assert torch.equal(gq, xq[ri]) and torch.equal(gs.view(torch.int32), xs[ri].view(torch.int32))


ACT_SHAPES = [(1, 128), (3, 256), (7, 200), (5, 300), (128, 512), (33, 4096), (2, 8), (9, 1000),
              (0, 128), (4, 0), (1, 12288), (300, 768)]


@pytest.mark.parametrize("m,k", ACT_SHAPES)
def test_act_quant_bit_exact(W, m, k):
    x = synth.activations(m, k, seed=m * 7919 + k, device="cpu")
    xb = synth.bf16_bits(x)
    xq, xs = W.quantize_act_per_token_group(x.cuda())
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_act_per_token_group(xb)
    assert (f32(xs).view(np.uint32) == s_ref.view(np.uint32)).all()
    assert (u8(xq) == q_ref).all()


def test_act_quant_every_bf16_value_against_several_scales(W):
    """Every finite BF16 bit pattern, in groups whose amax is fixed by one
    planted element: drives both the fast quotient path and its exact
    fallback near E4M3 rounding midpoints."""
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = (pats.astype(np.uint32) << 16).view(np.float32)
    pats = pats[np.isfinite(f)]
    for amax in [448.0, 1.0, 3.0, 0.0173, 1e-30, 3e38, 5.5e3, 1e-39, 2e-41]:
        keep = np.abs((pats.astype(np.uint32) << 16).view(np.float32)) <= amax
        vals = pats[keep]
        per = 127
        n = -(-len(vals) // per)
        grid = np.zeros((n, 128), np.uint16)
        padded = np.concatenate([vals, np.zeros(n * per - len(vals), np.uint16)])
        grid[:, :per] = padded.reshape(n, per)
        amax_bits = np.float32(amax).view(np.uint32) >> 16
        grid[:, per] = amax_bits  # BF16 truncation of amax: still >= every value
        got_q, got_s = W.quantize_act_per_token_group(_bf16_dev(grid))
        torch.cuda.synchronize()
        q_ref, s_ref = O.quantize_act_per_token_group(grid)
        assert (f32(got_s).view(np.uint32) == s_ref.view(np.uint32)).all(), amax
        assert (u8(got_q) == q_ref).all(), amax


def test_act_quant_zero_rows_and_signed_zero(W):
    x = np.zeros((4, 256), np.uint16)
    x[1, :] = 0x8000  # -0.0
    x[2, 5] = 0x3F80  # 1.0
    xq, xs = W.quantize_act_per_token_group(_bf16_dev(x))
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_act_per_token_group(x)
    assert (u8(xq) == q_ref).all() and (f32(xs) == s_ref).all()
    assert (u8(xq)[1] == 0x80).all() and f32(xs)[0, 0] == 1.0


# ------------------------------------------------------ weight quantizer

W_SHAPES = [(256, 512), (200, 392), (200, 300), (1, 8), (130, 136), (128, 128), (513, 1024),
            (7, 12288), (0, 4096), (384, 2048)]


@pytest.mark.parametrize("n,k", W_SHAPES)
def test_weight_quant_bit_exact(W, n, k):
    w = synth.weights(n, k, seed=n * 31 + k, device="cpu")
    if n * k:
        w.view(-1)[::997] *= 40  # some large entries so blocks differ in scale
    wb = synth.bf16_bits(w)
    wq, ws = W.quantize_weight_blockwise(w.cuda())
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_weight_blockwise(wb)
    assert (f32(ws).view(np.uint32) == s_ref.view(np.uint32)).all()
    assert (u8(wq) == q_ref).all()


def test_weight_quant_batched_matches_single(W):
    shapes = [(256, 512), (200, 392), (200, 300), (1, 8), (384, 1024), (0, 128)]
    ws_in = [synth.weights(n, k, seed=i, device="cuda") for i, (n, k) in enumerate(shapes)]
    outs = W.quantize_weight_blockwise_batched(ws_in)
    torch.cuda.synchronize()
    for w, (q, s) in zip(ws_in, outs):
        q_ref, s_ref = O.quantize_weight_blockwise(synth.bf16_bits(w))
        assert (u8(q) == q_ref).all() and (f32(s).view(np.uint32) == s_ref.view(np.uint32)).all()


def test_weight_quant_zero_block(W):
    w = np.zeros((256, 256), np.uint16)
    w[128:, 128:] = 0x3C00  # 2^-7 in one block only
    w[:128, 128:] = 0x8000  # -0.0 block
    wq, ws = W.quantize_weight_blockwise(_bf16_dev(w))
    torch.cuda.synchronize()
    q_ref, s_ref = O.quantize_weight_blockwise(w)
    assert (u8(wq) == q_ref).all() and (f32(ws) == s_ref).all()
    assert f32(ws)[0, 0] == 1.0 and (u8(wq)[:128, 128:] == 0x80).all()


def test_weight_quant_full_model_sampled(W):
    """The whole Qwen3-8B weight sync (36 layers x 4 matrices, 6.9e9 elements)
    in the launch configuration the benchmark times, checked on sampled
    128x128 blocks (first, last and random ones of every matrix)."""
    layers = synth.QWEN3_8B_LAYERS
    mats, outs = [], []
    for l in range(layers):
        for j, (name, (n, k)) in enumerate(synth.QWEN3_8B_LINEARS.items()):
            mats.append(synth.weights(n, k, seed=1000 * l + j, device="cuda"))
    outs = W.quantize_weight_blockwise_batched(mats)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    for idx in [0, 1, 2, 3, len(mats) - 4, len(mats) - 3, len(mats) - 2, len(mats) - 1] + list(
            rng.integers(0, len(mats), 6)):
        w = mats[idx]
        q, s = outs[idx]
        nbr, nbc = s.shape
        picks = [(0, 0), (nbr - 1, nbc - 1)] + [(int(rng.integers(nbr)), int(rng.integers(nbc))) for _ in range(6)]
        for bi, bj in picks:
            blk = w[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            q_ref, s_ref = O.quantize_weight_blockwise(synth.bf16_bits(blk))
            assert f32(s[bi, bj:bj + 1]).view(np.uint32)[0] == s_ref.view(np.uint32)[0, 0]
            assert (u8(q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]) == q_ref).all()
    del mats, outs
    torch.cuda.empty_cache()


# ----------------------------------------------------------- KV cache

@pytest.mark.parametrize("shape", [(2, 64, 8, 128), (1000003,), (5,), (3, 7)])
def test_kv_quant_bit_exact(W, shape):
    if len(shape) == 4:
        x = synth.kv_cache(seed=1, shape=shape, device="cpu")
    else:
        numel = int(np.prod(shape))
        x = synth.activations(1, numel, seed=numel, device="cpu").reshape(shape)
    xb = synth.bf16_bits(x)
    q, scale, amax = W.kv_amax_quantize(x.cuda())
    torch.cuda.synchronize()
    q_ref, s_ref, a_ref = O.kv_amax_quantize(xb)
    assert f32(amax)[0] == a_ref
    assert f32(scale).view(np.uint32)[0] == np.float32(s_ref).view(np.uint32)
    assert (u8(q) == q_ref).all()


def test_kv_modes_and_zero_tensor(W):
    x = synth.kv_cache(seed=11, shape=(2, 16, 8, 128), device="cuda")
    xb = synth.bf16_bits(x)
    _, scale, amax = W.kv_amax_quantize(x, mode=W.KV_AMAX_ONLY)
    torch.cuda.synchronize()
    q_ref, s_ref, a_ref = O.kv_amax_quantize(xb)
    assert f32(amax)[0] == a_ref and f32(scale)[0] == s_ref
    # reuse a stale, smaller scale: elements past 448 must saturate
    stale = torch.tensor([s_ref / 3], dtype=torch.float32, device="cuda")
    q, _, _ = W.kv_amax_quantize(x, scale=stale, mode=W.KV_QUANT_ONLY)
    torch.cuda.synchronize()
    assert (u8(q) == O.quantize_with_scale(xb, f32(stale)[0])).all()
    z = torch.zeros(1000, dtype=torch.bfloat16, device="cuda")
    q, scale, amax = W.kv_amax_quantize(z)
    torch.cuda.synchronize()
    assert f32(scale)[0] == 1.0 and f32(amax)[0] == 0.0 and (u8(q) == 0).all()
    e = torch.zeros(0, dtype=torch.bfloat16, device="cuda")
    _, scale, amax = W.kv_amax_quantize(e)
    torch.cuda.synchronize()
    assert f32(scale)[0] == 1.0 and f32(amax)[0] == 0.0


def test_kv_full_size_sampled(W):
    """K and V at [32, 8192, 8, 128]: amax and scale over the full tensors,
    codes on a 2M-element sample."""
    rng = np.random.default_rng(1)
    for seed in (5, 6):
        x = synth.kv_cache(seed=seed, device="cuda")
        q, scale, amax = W.kv_amax_quantize(x)
        torch.cuda.synchronize()
        xb = synth.bf16_bits(x).reshape(-1)
        a_ref = O.amax_bf16(xb)
        s_ref = O.scale_from_amax(a_ref)
        assert f32(amax)[0] == a_ref and f32(scale)[0] == s_ref
        idx = np.concatenate([np.arange(4096), xb.size - 1 - np.arange(4096),
                              rng.integers(0, xb.size, 2_000_000)])
        got = u8(q).reshape(-1)[idx]
        assert (got == O.quantize_with_scale(xb[idx], s_ref)).all()
        del x, q
    torch.cuda.empty_cache()


# ------------------------------------------------------- power-of-two scales

@pytest.mark.parametrize("m,k", [(1, 128), (7, 200), (128, 512), (33, 4096), (9, 1000), (2, 12)])
def test_act_quant_pow2_bit_exact(W, m, k):
    x = synth.activations(m, k, seed=m * 31 + k + 5, device="cpu")
    xq, xs = W.quantize_act_per_token_group(x.cuda(), pow2=True)
    q_ref, s_ref = O.quantize_blocks(synth.bf16_bits(x), 1, 128, pow2=True)
    assert (u8(xq) == q_ref).all()
    assert (f32(xs).view(np.uint32) == s_ref.view(np.uint32)).all()


@pytest.mark.parametrize("n,k", [(256, 512), (300, 200), (129, 1000), (6144, 4096), (5, 12)])
def test_weight_quant_pow2_bit_exact(W, n, k):
    w = synth.weights(n, k, seed=n + k, device="cpu")
    wq, ws = W.quantize_weight_blockwise(w.cuda(), pow2=True)
    q_ref, s_ref = O.quantize_blocks(synth.bf16_bits(w), 128, 128, pow2=True)
    assert (u8(wq) == q_ref).all()
    assert (f32(ws).view(np.uint32) == s_ref.view(np.uint32)).all()


def test_pow2_scales_extreme_magnitudes(W):
    """Groups spanning the BF16 range: subnormal groups (S down to 2^-141),
    all-zero groups (S = 1) and groups near the BF16 maximum (S = 2^120)."""
    bits = np.zeros((4, 256), np.uint16)
    bits[0] = 0x0001                      # smallest BF16 subnormal everywhere
    bits[1, :128] = 0x7F7F                # BF16 max
    bits[1, 128:] = 0x8000                # -0 group
    bits[2] = np.arange(256, dtype=np.uint16) | 0x0100
    bits[3, ::2] = 0x3F80                 # 1.0 and zeros
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    xq, xs = W.quantize_act_per_token_group(x, pow2=True)
    q_ref, s_ref = O.quantize_blocks(bits, 1, 128, pow2=True)
    assert (u8(xq) == q_ref).all()
    assert (f32(xs).view(np.uint32) == s_ref.view(np.uint32)).all()


def test_weight_quant_batched_pow2_matches_single(W):
    ws_ = [synth.weights(n, k, seed=40 + n, device="cuda") for n, k in [(256, 512), (300, 200), (128, 4096)]]
    outs = W.quantize_weight_blockwise_batched(ws_, pow2=True)
    for w, (q, s) in zip(ws_, outs):
        q1, s1 = W.quantize_weight_blockwise(w, pow2=True)
        assert torch.equal(q, q1) and torch.equal(s.view(torch.int32), s1.view(torch.int32))
