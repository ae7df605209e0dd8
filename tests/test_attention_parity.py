"""GPU parity of the FP8 decode attention against the oracle's FP64
attention: every output within 1e-3 * sv * sum_t p_t |dec(v_t)| plus half a
BF16 ulp (the documented accuracy), and within a much tighter 2^-14 of the
same sum, which binary32 accumulation reaches."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from parity_util import bf16_to_f64, bits16, ulp_bf16
from w8a8_gemm_rl_gb300 import synth

pytestmark = pytest.mark.gpu


def _codes(shape, g):
    c = torch.randint(0, 256, shape, generator=g, dtype=torch.int32)
    c[(c & 0x7F) == 0x7F] = 0x7E
    return c.to(torch.uint8)


def _check(out, ref, ab, rel, dropped=0.0):
    """dropped: the bound on the weights too small for f16 (below 2^-39 of
    the row's largest), which the kernels leave out."""
    got = bf16_to_f64(bits16(out)).reshape(ref.shape)
    err = np.abs(got - ref)
    bound = rel * ab + 0.5 * ulp_bf16(ref) + dropped
    bad = err > bound
    assert not bad.any(), (int(bad.sum()), float((err - bound).max()))


CASES = [  # batch, max_seq, q heads, kv heads, lengths
    (2, 300, 8, 2, [300, 123]), (3, 64, 4, 4, [1, 64, 0]), (2, 40, 4, 2, [40, 17]),
    (1, 1000, 32, 8, [997]), (2, 96, 16, 2, [96, 95]), (4, 7, 8, 8, [7, 1, 2, 3]),
    # 320 (sequence, KV head) slices: enough that each slice is split over
    # only 2 CTAs; ragged lengths from 0 to 64
    (40, 64, 32, 8, [(7 * i) % 65 for i in range(40)]),
    # 8 query heads per KV head: one CTA covers all 8 used MMA rows
    (3, 200, 64, 8, [200, 77, 1]),
    # 64 slices: each split over 4 CTAs
    (8, 100, 32, 8, [100, 99, 64, 33, 32, 31, 17, 0])]


@pytest.mark.parametrize("B,S,Hq,Hkv,lens", CASES)
def test_decode_attention_matches_oracle(W, B, S, Hq, Hkv, lens):
    g = torch.Generator().manual_seed(B * 1000 + S)
    q, k, v = _codes((B, Hq, 128), g), _codes((B, S, Hkv, 128), g), _codes((B, S, Hkv, 128), g)
    scales = torch.tensor([0.02, 0.03, 0.5], dtype=torch.float32)
    ln = torch.tensor(lens, dtype=torch.int32)
    dev = lambda t: t.cuda()
    out = W.fp8_decode_attention(dev(q), dev(scales[0:1]), dev(k), dev(scales[1:2]), dev(v),
                                 dev(scales[2:3]), dev(ln))
    torch.cuda.synchronize()
    ref, ab = O.decode_attention(q.numpy(), scales[0].item(), k.numpy(), scales[1].item(), v.numpy(),
                                 scales[2].item(), ln.numpy(), 1 / math.sqrt(128))
    _check(out, ref, ab, 1e-3)
    _check(out, ref, ab, 2.0 ** -14)
    for b, L in enumerate(lens):
        if L == 0:
            assert (bits16(out[b]) == 0).all()


def test_decode_attention_over_the_quantized_kv_cache(W):
    """The KV-cache layout of the recalibration step: K and V quantized by
    kv_amax_quantize ([4, 512, 8, 128], gains per channel), a query
    quantized per tensor, ragged lengths; 32 query heads over 8 KV heads."""
    kc = synth.kv_cache(seed=11, shape=(4, 512, 8, 128), device="cuda")
    vc = synth.kv_cache(seed=12, shape=(4, 512, 8, 128), device="cuda")
    qx = synth.kv_cache(seed=13, shape=(4, 32, 1, 128), device="cuda").reshape(4, 32, 128)
    kq, ks, _ = W.kv_amax_quantize(kc)
    vq, vs, _ = W.kv_amax_quantize(vc)
    qq, qs, _ = W.kv_amax_quantize(qx)
    ln = torch.tensor([512, 300, 1, 77], dtype=torch.int32, device="cuda")
    out = W.fp8_decode_attention(qq, qs, kq, ks, vq, vs, ln)
    torch.cuda.synchronize()
    ref, ab = O.decode_attention(qq.cpu().numpy(), qs.item(), kq.cpu().numpy(), ks.item(),
                                 vq.cpu().numpy(), vs.item(), ln.cpu().numpy(), 1 / math.sqrt(128))
    _check(out, ref, ab, 2.0 ** -14)


def test_decode_attention_full_cache_sampled(W):
    """The KV configuration itself ([32, 8192, 8, 128], 32 query heads):
    every output of two sequences (one full, one of 4097 tokens) against the
    oracle."""
    g = torch.Generator().manual_seed(7)
    B, S = 32, 8192
    k = _codes((B, S, 8, 128), g).cuda()
    v = _codes((B, S, 8, 128), g).cuda()
    q = _codes((B, 32, 128), g).cuda()
    sc = torch.tensor([0.01, 0.01, 0.25], dtype=torch.float32, device="cuda")
    ln = torch.full((B,), S, dtype=torch.int32, device="cuda")
    ln[5] = 4097
    out = W.fp8_decode_attention(q, sc[0:1], k, sc[1:2], v, sc[2:3], ln)
    torch.cuda.synchronize()
    for b in (5, 31):
        ref, ab = O.decode_attention(q[b:b + 1].cpu().numpy(), 0.01, k[b:b + 1].cpu().numpy(), 0.01,
                                     v[b:b + 1].cpu().numpy(), 0.25, ln[b:b + 1].cpu().numpy(),
                                     1 / math.sqrt(128))
        _check(out[b:b + 1], ref, ab, 2.0 ** -14)


def test_decode_attention_clamps_device_lengths(W):
    """Lengths are device data the host cannot check: the kernel clamps them
    to [0, max_seq], so a negative length gives zeros and one past max_seq
    attends to the whole sequence (the oracle run with the clamped lengths)."""
    g = torch.Generator().manual_seed(77)
    B, S, Hq, Hkv = 3, 50, 8, 2
    q, k, v = _codes((B, Hq, 128), g), _codes((B, S, Hkv, 128), g), _codes((B, S, Hkv, 128), g)
    scales = torch.tensor([0.02, 0.03, 0.5], dtype=torch.float32)
    ln = torch.tensor([-5, S + 100, 20], dtype=torch.int32)
    dev = lambda t: t.cuda()
    out = W.fp8_decode_attention(dev(q), dev(scales[0:1]), dev(k), dev(scales[1:2]), dev(v),
                                 dev(scales[2:3]), dev(ln))
    torch.cuda.synchronize()
    clamped = np.array([0, S, 20], np.int32)
    ref, ab = O.decode_attention(q.numpy(), scales[0].item(), k.numpy(), scales[1].item(), v.numpy(),
                                 scales[2].item(), clamped, 1 / math.sqrt(128))
    _check(out, ref, ab, 2.0 ** -14)
    assert (bits16(out[0]) == 0).all()


# ------------------------------------------------------------------ prefill

def _dropped_bound(v, sv, hq):
    """sv * 2^-39 * sum over keys j <= i of max_d |dec(v_j)|, per [b, i, h, 1]:
    the most that weights below 2^-39 of a row's largest can carry."""
    dv = np.abs(O.e4m3_decode(v)).max(axis=3)           # [B, S, Hkv]
    cum = np.cumsum(dv, axis=1)                          # keys 0..i
    cum = np.repeat(cum, hq // v.shape[2], axis=2)       # query head h reads KV head h // g
    return abs(sv) * 2.0 ** -39 * cum[..., None]

PREFILL_CASES = [  # batch, tokens per sequence, q heads, kv heads
    (1, 1, 4, 4), (2, 63, 8, 2), (1, 64, 4, 1), (2, 65, 4, 4), (1, 128, 4, 2), (2, 129, 8, 8),
    (1, 200, 8, 2), (1, 256, 4, 4), (3, 130, 32, 8), (1, 700, 8, 8),
    (2, 520, 16, 4)]  # 160 query blocks: some CTAs take two


@pytest.mark.parametrize("B,S,Hq,Hkv", PREFILL_CASES)
def test_prefill_attention_matches_oracle(W, B, S, Hq, Hkv):
    """Causal prefill over random E4M3 codes (every finite code): a single
    token, partial and whole 128-token query blocks and key chunks, grouped
    heads, more query blocks than SMs (a persistent CTA takes several)."""
    g = torch.Generator().manual_seed(B * 100 + S + Hq)
    q, k, v = _codes((B, S, Hq, 128), g), _codes((B, S, Hkv, 128), g), _codes((B, S, Hkv, 128), g)
    scales = torch.tensor([0.02, 0.03, 0.5], dtype=torch.float32)
    dev = lambda t: t.cuda()
    out = W.fp8_prefill_attention(dev(q), dev(scales[0:1]), dev(k), dev(scales[1:2]), dev(v),
                                  dev(scales[2:3]))
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    ref, ab = O.prefill_attention(q.numpy(), scales[0].item(), k.numpy(), scales[1].item(),
                                  v.numpy(), scales[2].item(), 1 / math.sqrt(128))
    drop = _dropped_bound(v.numpy(), scales[2].item(), Hq)
    _check(out, ref, ab, 1e-3, drop)
    _check(out, ref, ab, 2.0 ** -14, drop)


def test_prefill_attention_over_quantized_activations(W):
    """Q, K and V from N(0, 1) activations with 0.1% x50 outliers, each
    quantized per tensor by kv_amax_quantize (as the rollout stores them):
    the softmax is not dominated by a few keys here."""
    B, S, Hq, Hkv = 2, 300, 16, 4
    x = [synth.activations(B * S * h, 128, seed=90 + i).reshape(B, S, h, 128).cuda()
         for i, h in enumerate((Hq, Hkv, Hkv))]
    qkv = [W.kv_amax_quantize(t) for t in x]
    out = W.fp8_prefill_attention(qkv[0][0], qkv[0][1], qkv[1][0], qkv[1][1], qkv[2][0], qkv[2][1])
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    sc = [t[1].item() for t in qkv]
    ref, ab = O.prefill_attention(qkv[0][0].cpu().numpy(), sc[0], qkv[1][0].cpu().numpy(), sc[1],
                                  qkv[2][0].cpu().numpy(), sc[2], 1 / math.sqrt(128))
    drop = _dropped_bound(qkv[2][0].cpu().numpy(), sc[2], Hq)
    _check(out, ref, ab, 1e-3, drop)
    _check(out, ref, ab, 2.0 ** -14, drop)


def test_prefill_attention_full_size_sampled(W):
    """The bench's workload and launch: 4 sequences x 2048 tokens, 32 query
    heads over 8 KV heads, Q, K and V per-tensor-quantized N(0, 1)
    activations with outliers (the same seeds).  The oracle computes sampled
    (sequence, query head) slices one by one: first and last, and heads of
    different KV groups."""
    B, S, Hq, Hkv = 4, 2048, 32, 8
    x = [synth.activations(B * S * h, 128, seed=95 + i, device="cuda").reshape(B, S, h, 128)
         for i, h in enumerate((Hq, Hkv, Hkv))]
    qkv = [W.kv_amax_quantize(t) for t in x]
    out = W.fp8_prefill_attention(qkv[0][0], qkv[0][1], qkv[1][0], qkv[1][1], qkv[2][0], qkv[2][1])
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    sc = [t[1].item() for t in qkv]
    q, k, v = (t[0].cpu().numpy() for t in qkv)
    for b, h in [(0, 0), (1, 13), (2, 22), (3, 31)]:
        kh = h // (Hq // Hkv)
        qs, ks, vs = (np.ascontiguousarray(a[b:b + 1, :, j:j + 1]) for a, j in ((q, h), (k, kh), (v, kh)))
        ref, ab = O.prefill_attention(qs, sc[0], ks, sc[1], vs, sc[2], 1 / math.sqrt(128))
        drop = _dropped_bound(vs, sc[2], 1)
        got = out[b:b + 1, :, h:h + 1].contiguous()
        _check(got, ref, ab, 1e-3, drop)
        _check(got, ref, ab, 2.0 ** -14, drop)
