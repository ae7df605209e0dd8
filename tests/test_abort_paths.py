"""The kernels' abort paths, run on demand: with the test hook on, a bounded
wait behaves as if it had run out of time.  The kernel must return (no
hang), report the documented code through w8a8_consume_device_error, and
leave the GPU usable: the next normal call passes parity.  Nothing here
faults or hangs a GPU: the hook only makes one wait give up early."""
import numpy as np
import pytest
import torch

import math

import oracle as O
from parity_util import assert_gemm_close, bf16_to_f64, bits16, ulp_bf16
from w8a8_gemm_rl_gb300 import synth

pytestmark = pytest.mark.gpu


def _gemm_case(m, n, k, seed):
    g = torch.Generator().manual_seed(seed)
    xq = (torch.randn(m, k, generator=g) * 60).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    wq = (torch.randn(n, k, generator=g) * 60).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    xs = (torch.rand(m, -(-k // 128), generator=g) * 0.01 + 0.001).numpy()
    ws = (torch.rand(-(-n // 128), -(-k // 128), generator=g) * 0.01 + 0.001).numpy()
    return xq, xs, wq, ws


@pytest.mark.parametrize("m,code", [(300, 5), (64, 35)])
def test_gemm_abort_then_recover(W, m, code):
    n, k = 512, 1024
    xq, xs, wq, ws = _gemm_case(m, n, k, seed=m)
    dev = [torch.from_numpy(a).cuda() for a in (xq, xs, wq, ws)]
    assert W.consume_device_error() == 0
    W.debug_force_wait_timeout(True)
    try:
        W.fp8_block_gemm(*dev)
        torch.cuda.synchronize()
    finally:
        W.debug_force_wait_timeout(False)
    assert W.consume_device_error() == code
    y = W.fp8_block_gemm(*dev)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    y_ref, absref = O.block_gemm(xq, xs, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, f"after abort m={m}")


def test_pow2_gemm_abort_then_recover(W):
    m, n, k = 300, 512, 1024
    xq, _, wq, _ = _gemm_case(m, n, k, seed=17)
    rng = np.random.default_rng(17)
    xs = np.ldexp(np.float32(1), rng.integers(-12, -4, (m, k // 128))).astype(np.float32)
    ws = np.ldexp(np.float32(1), rng.integers(-12, -4, (n // 128, k // 128))).astype(np.float32)
    dev = [torch.from_numpy(a).cuda() for a in (xq, xs, wq, ws)]
    assert W.consume_device_error() == 0
    W.debug_force_wait_timeout(True)
    try:
        W.fp8_block_gemm_pow2(*dev)
        torch.cuda.synchronize()
    finally:
        W.debug_force_wait_timeout(False)
    assert W.consume_device_error() == 55
    y = W.fp8_block_gemm_pow2(*dev)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    y_ref, absref = O.block_gemm(xq, xs, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, "pow2 after abort")


def test_grouped_gemm_abort_then_recover(W):
    g, n, k, rows = 4, 256, 512, 200
    xq, xs, _, _ = _gemm_case(rows, n, k, seed=9)
    rng = np.random.default_rng(9)
    wq = np.stack([_gemm_case(1, n, k, seed=20 + e)[2] for e in range(g)])
    ws = np.stack([_gemm_case(1, n, k, seed=30 + e)[3] for e in range(g)])
    off = np.array([0, 37, 37, 120, rows], np.int32)
    ridx = rng.integers(0, rows, rows).astype(np.int32)
    args = [torch.from_numpy(xq).cuda(), torch.from_numpy(xs).cuda(), torch.from_numpy(ridx).cuda(),
            torch.from_numpy(off).cuda(), rows, torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda()]
    W.debug_force_wait_timeout(True)
    try:
        W.fp8_grouped_gemm(*args)
        torch.cuda.synchronize()
    finally:
        W.debug_force_wait_timeout(False)
    assert W.consume_device_error() == 5
    y = W.fp8_grouped_gemm(*args)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    y_ref, absref = O.grouped_gemm(xq, xs, ridx, off, wq, ws)
    assert_gemm_close(bits16(y), y_ref, absref, "grouped after abort")


def test_weight_quant_abort_then_recover(W):
    w = synth.weights(384, 1024, seed=5)
    W.debug_force_wait_timeout(True)
    try:
        W.quantize_weight_blockwise(w.cuda())
        torch.cuda.synchronize()   # the producer gives up on its own bounded wait (2 s)
    finally:
        W.debug_force_wait_timeout(False)
    assert W.consume_device_error() in (13, 11)
    wq, ws = W.quantize_weight_blockwise(w.cuda())
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    wq_ref, ws_ref = O.quantize_weight_blockwise(synth.bf16_bits(w))
    assert (wq.cpu().numpy() == wq_ref).all() and (ws.cpu().numpy() == ws_ref).all()


def _attention_case(B, S, Hq, Hkv, seed, query_tokens):
    g = torch.Generator().manual_seed(seed)

    def codes(shape):
        c = torch.randint(0, 256, shape, generator=g, dtype=torch.int32)
        c[(c & 0x7F) == 0x7F] = 0x7E  # every finite E4M3 code
        return c.to(torch.uint8)

    q = codes((B, S, Hq, 128) if query_tokens else (B, Hq, 128))
    return q, codes((B, S, Hkv, 128)), codes((B, S, Hkv, 128)), [0.02, 0.03, 0.5]


def _attention_close(out, ref, ab, dropped):
    """The documented accuracy: 1e-3 * sv * sum p |dec(v)| plus half a BF16
    ulp plus what the weights f16 cannot hold (below 2^-39 of a row's
    largest) can carry."""
    got = bf16_to_f64(bits16(out)).reshape(ref.shape)
    bad = np.abs(got - ref) > 1e-3 * ab + 0.5 * ulp_bf16(ref) + dropped
    assert not bad.any(), int(bad.sum())


def _vmax(v):
    return np.abs(O.e4m3_decode(v.numpy())).max(axis=3)  # [B, S, Hkv]


def test_decode_attention_abort_then_recover(W):
    q, k, v, sc = _attention_case(2, 300, 8, 2, seed=21, query_tokens=False)
    lens = torch.tensor([300, 123], dtype=torch.int32)
    dev = [t.cuda() for t in (q, k, v, lens)] + [torch.tensor([x]).cuda() for x in sc]
    args = (dev[0], dev[4], dev[1], dev[5], dev[2], dev[6], dev[3])
    assert W.consume_device_error() == 0
    W.debug_force_wait_timeout(True)
    try:
        W.fp8_decode_attention(*args)
        torch.cuda.synchronize()
    finally:
        W.debug_force_wait_timeout(False)
    assert W.consume_device_error() == 21
    out = W.fp8_decode_attention(*args)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    ref, ab = O.decode_attention(q.numpy(), sc[0], k.numpy(), sc[1], v.numpy(), sc[2],
                                 lens.numpy(), 1 / math.sqrt(128))
    vm = _vmax(v)
    per_bh = np.stack([vm[b, :L].sum(axis=0) for b, L in enumerate(lens.tolist())])  # [B, Hkv]
    dropped = sc[2] * 2.0 ** -39 * np.repeat(per_bh, 4, axis=1)[..., None]  # [B, Hq, 1]
    _attention_close(out, ref, ab, dropped)


def test_prefill_attention_abort_then_recover(W):
    q, k, v, sc = _attention_case(2, 300, 8, 2, seed=23, query_tokens=True)
    dev = [t.cuda() for t in (q, k, v)] + [torch.tensor([x]).cuda() for x in sc]
    args = (dev[0], dev[3], dev[1], dev[4], dev[2], dev[5])
    assert W.consume_device_error() == 0
    W.debug_force_wait_timeout(True)
    try:
        W.fp8_prefill_attention(*args)
        torch.cuda.synchronize()
    finally:
        W.debug_force_wait_timeout(False)
    assert W.consume_device_error() == 23
    out = W.fp8_prefill_attention(*args)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    ref, ab = O.prefill_attention(q.numpy(), sc[0], k.numpy(), sc[1], v.numpy(), sc[2],
                                  1 / math.sqrt(128))
    cum = np.repeat(np.cumsum(_vmax(v), axis=1), 4, axis=2)  # keys 0..i, per query head
    _attention_close(out, ref, ab, sc[2] * 2.0 ** -39 * cum[..., None])
