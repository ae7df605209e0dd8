"""Pins for the CPU oracle, checked against things other than the oracle itself:
the values the pages print (E4M3 range +-448), the OCP format facts they cite,
hand-worked roundings, a library codec (torch float8_e4m3fn), a second encoder
written differently, closed forms, invariants and brute force on tiny inputs.
CPU only."""
import math
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_encode(x32):
    """Library encode, valid for |x| <= 448 (torch does not saturate)."""
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()[:2]
            rows.append((a, b))
    return rows


# ---------------------------------------------------------------- E4M3 codec

def test_decode_landmarks_from_pages_and_spec():
    for code, val in _read_table("e4m3_landmarks.txt"):
        got = O.lib().oracle_e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val), code
            assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_decode_matches_library_codec_all_256():
    ours = O.e4m3_decode(np.arange(256))
    lib = _torch_decode_all()
    nan = np.isnan(lib)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == lib[~nan]).all()
    assert (np.signbit(ours[~nan]) == np.signbit(lib[~nan])).all()
    assert np.nanmax(ours) == 448.0 and np.nanmin(ours) == -448.0


def test_encode_roundtrip_254_codes():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = O.lib().oracle_e4m3_decode(c)
        assert O.e4m3_encode_scalar(v) == c, hex(c)
        assert O.e4m3_encode_bits_scalar(v) == c, hex(c)


def test_encode_hand_rounding():
    for x, code in _read_table("e4m3_hand_rounding.txt"):
        v = float(np.float32(float(x)))
        assert O.e4m3_encode_scalar(v) == int(code, 16), x
        assert O.e4m3_encode_bits_scalar(v) == int(code, 16), x


def _band_check(args):
    start, count = args
    import oracle as O2
    return O2.e4m3_cross_check(start, count)


def test_encoders_agree_exhaustive_band():
    """Encoder A (grid search) vs encoder B (bit fields) on every positive
    binary32 in [2^-12, 512), where all the rounding decisions are, and on a
    stride through everything else (both signs, NaNs skipped)."""
    lo = np.float32(2.0 ** -12).view(np.uint32).item()
    hi = np.float32(512.0).view(np.uint32).item()
    chunk = 1 << 22
    jobs = [(s, min(chunk, hi - s)) for s in range(lo, hi, chunk)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(8, os.cpu_count() or 1)) as pool:
        res = pool.map(_band_check, jobs)
    bad = sum(r[0] for r in res)
    assert bad == 0, [r for r in res if r[0]][:3]
    # everything else: 4096-pattern windows spread over all 2^32 patterns
    for off in range(0, 1 << 32, 1 << 22):
        b, first = O.e4m3_cross_check(off, 4096)
        assert b == 0, hex(first)


def test_encoder_matches_library_in_range():
    """Against torch's float8_e4m3fn conversion for |x| <= 448: every E4M3
    rounding midpoint and its +-3 ulp neighbours, plus a dense random sample."""
    grid = O.e4m3_decode(np.arange(0, 127))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)  # exact in binary32
    assert (mids.astype(np.float64) == (grid[:-1] + grid[1:]) / 2).all()
    bits = mids.view(np.uint32).astype(np.int64)
    near = (bits[:, None] + np.arange(-3, 4)[None, :]).reshape(-1).astype(np.uint32)
    rng = np.random.default_rng(0)
    rand = (rng.standard_normal(2_000_000) * rng.choice([1e-3, 1e-1, 1, 30, 200], 2_000_000))
    x = np.concatenate([near.view(np.float32), rand.astype(np.float32), grid.astype(np.float32)])
    x = np.concatenate([x, -x])
    x = x[np.abs(x) <= 448]
    assert (O.e4m3_encode(x) == _torch_encode(x)).all()


def test_encode_monotone_and_saturating():
    x = np.sort(np.random.default_rng(1).uniform(-600, 600, 500_000).astype(np.float32))
    v = O.e4m3_decode(O.e4m3_encode(x))
    assert (np.diff(v) >= 0).all()
    assert v.max() == 448 and v.min() == -448
    assert (O.e4m3_encode(np.array([np.inf, -np.inf], np.float32)) == [0x7E, 0xFE]).all()


# ------------------------------------------------------------------- scales

def test_scale_closed_forms():
    assert O.scale_from_amax(448.0) == 1.0
    assert O.scale_from_amax(896.0) == 2.0
    assert O.scale_from_amax(0.0) == 1.0
    assert O.scale_from_amax(3.5) == np.float32(3.5) / np.float32(448.0)
    amax = np.abs(np.random.default_rng(2).standard_normal(10000)).astype(np.float32) * 100
    s = np.array([O.scale_from_amax(a) for a in amax], np.float32)
    back = (s.astype(np.float64) * 448.0)
    ulp = np.spacing(amax).astype(np.float64)
    assert (np.abs(back - amax) <= ulp).all()


# --------------------------------------------------------------- quantizers

def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _library_quantize(xbits, br, bc):
    """The quantizer restated with library routines only: numpy for amax and
    the binary32 division, torch float8_e4m3fn for the rounding (after the
    saturation the pages' range implies)."""
    x = _f32(xbits)
    rows, cols = x.shape
    nbr, nbc = -(-rows // br), -(-cols // bc)
    q = np.zeros((rows, cols), np.uint8)
    s = np.zeros((nbr, nbc), np.float32)
    for bi in range(nbr):
        for bj in range(nbc):
            blk = x[bi * br:(bi + 1) * br, bj * bc:(bj + 1) * bc]
            amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
            sc = np.float32(1) if amax == 0 else np.float32(amax / np.float32(448))
            s[bi, bj] = sc
            t = (blk / sc).astype(np.float32)
            t = np.clip(t, -448, 448)
            q[bi * br:(bi + 1) * br, bj * bc:(bj + 1) * bc] = _torch_encode(t).reshape(blk.shape)
    return q, s


@pytest.mark.parametrize("shape,br,bc", [((256, 384), 128, 128), ((200, 300), 128, 128),
                                          ((7, 333), 1, 128), ((1, 1000), 1, 1000),
                                          ((130, 129), 128, 128), ((0, 5), 1, 128)])
def test_quantizer_matches_library_restatement(shape, br, bc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(shape).astype(np.float32)
    if x.size:
        x.reshape(-1)[rng.choice(x.size, max(1, x.size // 1000), replace=False)] *= 50
    xb = _bf16(x)
    q, s = O.quantize_blocks(xb, br, bc)
    q2, s2 = _library_quantize(xb, br, bc)
    assert (s == s2).all()
    assert (q == q2).all()


def test_hand_blocks_scale_one_and_two():
    rng = np.random.default_rng(4)
    w = rng.uniform(-400, 400, (128, 256)).astype(np.float32)
    w[5, 7] = 448.0     # block 0: amax 448 -> S = 1, q = enc(x)
    w[9, 200] = -896.0  # block 1: amax 896 -> S = 2, q = enc(x / 2) (exact halves)
    wb = _bf16(w)
    q, s = O.quantize_weight_blockwise(wb)
    assert s.tolist() == [[1.0, 2.0]]
    x = _f32(wb)
    assert (q[:, :128] == _torch_encode(x[:, :128])).all()
    assert (q[:, 128:] == _torch_encode(x[:, 128:] / 2)).all()
    assert q[5, 7] == 0x7E and q[9, 200] == 0xFE


def test_all_zero_block_and_signed_zero():
    x = np.zeros((128, 128), np.float32)
    x[3, :] = -0.0
    q, s = O.quantize_weight_blockwise(_bf16(x))
    assert s.tolist() == [[1.0]]
    assert (q[3] == 0x80).all() and (np.delete(q, 3, axis=0) == 0).all()


def test_quantizer_invariants():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 1024)) * rng.choice([1e-3, 1, 40], (64, 1))).astype(np.float32)
    xb = _bf16(x)
    xf = _f32(xb)
    q, s = O.quantize_act_per_token_group(xb)
    dec = O.e4m3_decode(q)
    for i in range(64):
        for g in range(8):
            cq = q[i, g * 128:(g + 1) * 128]
            assert (cq == 0x7E).any() or (cq == 0xFE).any()  # the amax element hits 448
            xs = xf[i, g * 128:(g + 1) * 128]
            order = np.argsort(xs, kind="stable")
            assert (np.diff(dec[i, g * 128:(g + 1) * 128][order]) >= 0).all()  # monotone
            # rounding error at most half an E4M3 spacing (relative 2^-4) of x/S,
            # or half the subnormal quantum 2^-10, plus binary32 division slack
            t = xs.astype(np.float64) / s[i, g]
            err = np.abs(dec[i, g * 128:(g + 1) * 128] - t)
            bound = np.maximum(np.abs(t) * 2.0 ** -4, 2.0 ** -10) * (1 + 2.0 ** -20)
            assert (err <= bound).all()


def test_gather_commutes_with_per_token_quant():
    rng = np.random.default_rng(6)
    xb = _bf16(rng.standard_normal((50, 384)))
    idx = rng.integers(0, 50, 120)
    q1, s1 = O.quantize_act_per_token_group(xb)
    q2, s2 = O.quantize_act_per_token_group(xb[idx])
    assert (q1[idx] == q2).all() and (s1[idx] == s2).all()


def test_routed_row_quant_is_quant_then_gather_with_zero_rows():
    """The routed-row quantizer of the oracle: valid indices give the rows of
    the plain per-token quantization (quantization works per row), duplicated
    indices identical rows, and an index outside [0, rows_x) the quantization
    of an all-zero row: codes 0x00, scale 1 (the all-zero group's reading)."""
    rng = np.random.default_rng(16)
    xb = _bf16(rng.standard_normal((40, 384)) * 3.0)
    idx = np.concatenate([rng.integers(0, 40, 90), [-1, 40, 7, 7, 2 ** 31 - 1, -(2 ** 31)]])
    q, s = O.quantize_act_per_token_group_gather(xb, idx)
    qd, sd = O.quantize_act_per_token_group(xb)
    ok = (idx >= 0) & (idx < 40)
    assert (q[ok] == qd[idx[ok]]).all() and (s[ok] == sd[idx[ok]]).all()
    assert (q[~ok] == 0).all() and (s[~ok] == 1.0).all()
    assert (q[-4] == q[-3]).all()
    # and not the identity: a shifted index set changes the rows
    q2, _ = O.quantize_act_per_token_group_gather(xb, (idx[ok] + 1) % 40)
    assert (q2 != q[ok]).any()


# ------------------------------------------------- decode attention (FP8 KV)

def _attn_inputs(rng, B, S, Hq, Hkv, D=128):
    def codes(shape):
        c = rng.integers(0, 256, shape).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x7E
        return c
    return codes((B, Hq, D)), codes((B, S, Hkv, D)), codes((B, S, Hkv, D))


def test_attention_closed_forms():
    """One token: the output is that token's dequantized V.  A zero query:
    uniform weights, so the output is the mean of the dequantized V rows.
    No tokens: zeros.  Each query head reads KV head h / (Hq / Hkv)."""
    rng = np.random.default_rng(30)
    q, k, v = _attn_inputs(rng, 3, 20, 8, 2)
    sv = 0.375
    lens = np.array([1, 20, 0], np.int32)
    out, _ = O.decode_attention(q, 0.01, k, 0.02, v, sv, lens, 1 / np.sqrt(128))
    for h in range(8):
        assert np.array_equal(out[0, h], sv * O.e4m3_decode(v[0, 0, h // 4]))
    assert (out[2] == 0).all()
    qz = np.zeros_like(q)
    outz, _ = O.decode_attention(qz, 1.0, k, 1.0, v, sv, lens, 1.0)
    for h in range(8):
        want = sv * O.e4m3_decode(v[1, :20, h // 4]).mean(axis=0)
        assert np.allclose(outz[1, h], want, rtol=1e-14, atol=1e-300)
    # GQA: KV heads holding distinct constants show which one each query head read
    vc = np.zeros_like(v)
    vc[:, :, 0, :] = 0x38  # 1.0
    vc[:, :, 1, :] = 0x40  # 2.0
    outc, _ = O.decode_attention(q, 0.01, k, 0.02, vc, 1.0, lens, 1 / np.sqrt(128))
    assert (outc[1, :4] == 1.0).all() and (outc[1, 4:] == 2.0).all()


def test_attention_matches_library_softmax():
    """Against torch: float64 softmax and einsum over the dequantized
    tensors (library routines, written independently of the oracle)."""
    rng = np.random.default_rng(31)
    B, S, Hq, Hkv = 2, 37, 8, 2
    q, k, v = _attn_inputs(rng, B, S, Hq, Hkv)
    # the scales are binary32 values (as the library stores them)
    sq, sk, sv = (float(np.float32(t)) for t in (0.02, 0.05, 0.5))
    sc = 1 / np.sqrt(128)
    lens = np.array([37, 23], np.int32)
    out, ab = O.decode_attention(q, sq, k, sk, v, sv, lens, sc)
    dq = torch.from_numpy(O.e4m3_decode(q)) * sq
    dk = torch.from_numpy(O.e4m3_decode(k)) * sk
    dv = torch.from_numpy(O.e4m3_decode(v)) * sv
    for b in range(B):
        L = int(lens[b])
        kk = dk[b, :L].repeat_interleave(Hq // Hkv, dim=1)  # [L, Hq, D]
        vv = dv[b, :L].repeat_interleave(Hq // Hkv, dim=1)
        p = torch.softmax(torch.einsum("hd,thd->ht", dq[b], kk) * sc, dim=-1)
        want = torch.einsum("ht,thd->hd", p, vv).numpy()
        assert np.allclose(out[b], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
        assert (ab[b] >= np.abs(out[b]) * (1 - 1e-12)).all()


# ------------------------------------------------------ prefill attention

def test_prefill_attention_pins():
    """Causal prefill attention against what fixes it:
    * query token 0 has one key, so its output is that token's dequantized V;
    * a zero query weighs keys 0..i uniformly: the mean of those V rows;
    * query token S-1 sees the whole sequence: the (separately pinned) decode
      attention over all S tokens;
    * causality: changing K and V of tokens after i leaves row i unchanged;
    * grouped heads: Hkv = 2 KV heads give what Hkv = 8 with each KV head
      repeated for its 4 query heads gives."""
    rng = np.random.default_rng(40)
    B, S, Hq, Hkv = 2, 19, 8, 2
    qd, k, v = _attn_inputs(rng, B * S, S, Hq, Hkv)
    q = qd.reshape(B, S, Hq, 128)
    k, v = k[:B], v[:B]
    sq, sk, sv = (float(np.float32(t)) for t in (0.02, 0.05, 0.375))
    sc = 1 / np.sqrt(128)
    out, ab = O.prefill_attention(q, sq, k, sk, v, sv, sc)
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(out[b, 0, h], sv * O.e4m3_decode(v[b, 0, h // 4]))
    assert (ab >= np.abs(out) * (1 - 1e-12)).all()
    outz, _ = O.prefill_attention(np.zeros_like(q), 1.0, k, 1.0, v, sv, 1.0)
    for i in (0, 5, S - 1):
        for h in range(Hq):
            want = sv * O.e4m3_decode(v[1, : i + 1, h // 4]).mean(axis=0)
            assert np.allclose(outz[1, i, h], want, rtol=1e-14, atol=1e-300)
    lens = np.full(B, S, np.int32)
    dec, _ = O.decode_attention(np.ascontiguousarray(q[:, S - 1]), sq, k, sk, v, sv, lens, sc)
    assert np.allclose(out[:, S - 1], dec, rtol=1e-13, atol=1e-13 * np.abs(dec).max())
    i = 7
    k2, v2 = k.copy(), v.copy()
    k2[:, i + 1 :] = rng.integers(0, 0x7E, k2[:, i + 1 :].shape)
    v2[:, i + 1 :] = rng.integers(0, 0x7E, v2[:, i + 1 :].shape)
    out2, _ = O.prefill_attention(q, sq, k2, sk, v2, sv, sc)
    assert np.array_equal(out2[:, : i + 1], out[:, : i + 1])
    assert not np.array_equal(out2[:, i + 1 :], out[:, i + 1 :])
    out8, _ = O.prefill_attention(q, sq, np.repeat(k, 4, axis=2), sk, np.repeat(v, 4, axis=2), sv, sc)
    assert np.array_equal(out8, out)


def test_prefill_attention_matches_library_softmax():
    """Against torch: a float64 causal softmax (masked with -inf) and einsum
    over the dequantized tensors, library routines written independently."""
    rng = np.random.default_rng(41)
    B, S, Hq, Hkv = 2, 23, 4, 4
    qd, k, v = _attn_inputs(rng, B * S, S, Hq, Hkv)
    q = qd.reshape(B, S, Hq, 128)
    k, v = k[:B], v[:B]
    sq, sk, sv = (float(np.float32(t)) for t in (0.03, 0.04, 0.5))
    sc = 1 / np.sqrt(128)
    out, _ = O.prefill_attention(q, sq, k, sk, v, sv, sc)
    dq = torch.from_numpy(O.e4m3_decode(q)) * sq
    dk = torch.from_numpy(O.e4m3_decode(k)) * sk
    dv = torch.from_numpy(O.e4m3_decode(v)) * sv
    mask = torch.triu(torch.ones(S, S, dtype=torch.bool), diagonal=1)
    for b in range(B):
        s = torch.einsum("ihd,jhd->hij", dq[b], dk[b]) * sc
        p = torch.softmax(s.masked_fill(mask, float("-inf")), dim=-1)
        want = torch.einsum("hij,jhd->ihd", p, dv[b]).numpy()
        assert np.allclose(out[b], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


# ------------------------------------------------------ power-of-two scales

def test_pow2_scale_hand_values_and_definition():
    """S is the smallest power of two with 448 S >= amax: hand values at the
    boundaries (448 -> 1, 448 + 1 ulp -> 2, 224 -> 1/2, 1 -> 2^-8 since
    448 * 2^-9 = 0.875 < 1), the zero group, the extremes of BF16, and on a
    sweep: a power of two (frexp mantissa 1/2), 448 S >= amax, 448 S/2 < amax."""
    f32 = np.float32
    assert O.scale_pow2_from_amax(0.0) == 1.0
    assert O.scale_pow2_from_amax(448.0) == 1.0
    assert O.scale_pow2_from_amax(float(np.nextafter(f32(448), f32(1e9)))) == 2.0
    assert O.scale_pow2_from_amax(224.0) == 0.5 and O.scale_pow2_from_amax(1.0) == 2.0 ** -8
    assert O.scale_pow2_from_amax(2.0 ** -133) == 2.0 ** -141  # smallest BF16 subnormal
    assert O.scale_pow2_from_amax(float(_bf16_val(np.array([0x7F7F]))[0])) == 2.0 ** 120
    rng = np.random.default_rng(23)
    for a in np.exp(rng.uniform(-80, 80, 2000)).astype(np.float32):
        sc = O.scale_pow2_from_amax(float(a))
        m, _ = np.frexp(sc)
        assert m == 0.5 and 448.0 * sc >= a and 448.0 * sc / 2 < a


def test_pow2_quant_is_one_rounding_of_an_exact_quotient():
    """With S a power of two, x / S is exact, so a code is torch's E4M3
    rounding of x * 2^-e; no code saturates: amax / S lies in (224, 448], so
    the largest code magnitude in a non-zero group lies in [224, 448]
    (224 itself when amax / S rounds down to it, the grid step there being 32)."""
    rng = np.random.default_rng(24)
    xb = _bf16(rng.standard_normal((64, 384)) * np.where(rng.random((64, 384)) < 0.01, 50, 1))
    q, s = O.quantize_blocks(xb, 1, 128, pow2=True)
    x = _bf16_val(xb).astype(np.float32)
    S = np.repeat(s, 128, 1)
    t = torch.from_numpy((x / S).astype(np.float32))
    want = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (q == want).all()
    mag = np.abs(O.e4m3_decode(q)).reshape(64, 3, 128).max(-1)
    assert ((mag >= 224) & (mag <= 448)).all()


# ------------------------------------------------- dequantization (fake quant)

def _bf16_val(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_dequant_with_unit_scale_is_the_format_decode():
    """With S = 1 the dequantized BF16 value is the code's E4M3 value itself
    (every E4M3 value has at most 4 significant bits, so BF16 holds it):
    the landmarks of the format come back, and every non-NaN code decodes to
    the pinned decoder's value, signs included."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8).reshape(1, -1)
    y = _bf16_val(O.dequantize_blocks(codes, np.ones((1, 1), np.float32), 1, codes.shape[1]))[0]
    want = O.e4m3_decode(codes[0])
    assert (y == want).all() and (np.signbit(y) == np.signbit(want)).all()
    d = dict(zip(codes[0].tolist(), y.tolist()))
    assert d[0x7E] == 448.0 and d[0xFE] == -448.0 and d[0x01] == 2.0 ** -9 and d[0x38] == 1.0


def test_dequant_scales_by_powers_of_two_exactly():
    codes = np.arange(0, 0x7F, dtype=np.uint8).reshape(1, -1)
    base = _bf16_val(O.dequantize_blocks(codes, np.ones((1, 1), np.float32), 1, 127))
    for j in (-20, -3, 1, 7, 30):
        y = _bf16_val(O.dequantize_blocks(codes, np.full((1, 1), 2.0 ** j, np.float32), 1, 127))
        assert (y == base * 2.0 ** j).all()


def test_dequant_rounds_the_binary32_product_to_bf16():
    """Hand-worked double rounding (the reading: one binary32 multiply, then
    BF16 round-to-nearest-even).  For d = 1.125 (code 0x39) pick the binary32
    S whose exact product d*S lies just above 1 + 2^-8 (the midpoint between
    the BF16 neighbours 1 and 1 + 2^-7) but rounds to that midpoint in
    binary32; the tie then goes to the even BF16 value 1.0.  Rounding the
    exact product once would give 1 + 2^-7 instead."""
    d = 1.125
    found = None
    s = np.float32((1 + 2.0 ** -8) / d)
    for _ in range(64):
        exact = d * float(s)
        if exact > 1 + 2.0 ** -8 and float(np.float32(d) * s) == 1 + 2.0 ** -8:
            found = s
            break
        s = np.nextafter(s, np.float32(2.0))
    assert found is not None
    y = _bf16_val(O.dequantize_blocks(np.array([[0x39]], np.uint8), np.array([[found]], np.float32), 1, 1))
    assert y[0, 0] == 1.0


def test_dequant_of_quant_is_within_half_a_code_step():
    """Round trip: |BF16(dec(q) S) - x| <= (half an E4M3 spacing of x/S, or
    half the subnormal quantum) * S + half a BF16 ulp, on weights and on
    activations with outliers; a transposed or shifted scale grid fails it."""
    rng = np.random.default_rng(21)
    for (r, c, br, bc) in [(256, 384, 128, 128), (37, 300, 1, 128)]:
        xb = _bf16(rng.standard_normal((r, c)) * np.where(rng.random((r, c)) < 0.01, 50, 1))
        q, s = O.quantize_blocks(xb, br, bc)
        y = _bf16_val(O.dequantize_blocks(q, s, br, bc))
        x = _bf16_val(xb)
        S = np.repeat(np.repeat(s, br, 0), bc, 1)[:r, :c].astype(np.float64)
        t = np.abs(x) / S
        step = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(t, 2.0 ** -6))) - 3), 2.0 ** -9)
        bound = 0.5 * step * S * (1 + 2.0 ** -20) + 2.0 ** -8 * np.abs(y)
        assert (np.abs(y - x) <= bound).all()
        if br == 128 and s.shape[0] > 1 and s.shape[1] > 1:
            yt = _bf16_val(O.dequantize_blocks(q, np.ascontiguousarray(s[::-1]), br, bc))
            assert not (np.abs(yt - x) <= bound).all()


def test_quant_error_hand_block_and_library_sums():
    """A hand-worked block: amax 448 gives S = 1; 1.0625 lies halfway
    between the E4M3 values 1.0 and 1.125 and goes to 1.0, so e = 1/16:
    max 0.0625, sum e^2 = 2^-8, sum x^2 = 1 + 1.12890625 + 200704 + 9.
    Then random blocks: the sums equal numpy's float64 sums, and reporting
    over 1x128 or 128x128 blocks gives the same totals."""
    xb = _bf16(np.array([[1.0, 1.0625, 448.0, 3.0]]))
    q, s = O.quantize_blocks(xb, 1, 4)
    assert s[0, 0] == 1.0
    st = O.quant_error(xb, q, s, 1, 4, 1, 4)[0, 0]
    assert st[0] == 0.0625 and st[1] == 2.0 ** -8 and st[2] == 1 + 1.12890625 + 200704 + 9
    rng = np.random.default_rng(22)
    xb = _bf16(rng.standard_normal((256, 384)))
    q, s = O.quantize_blocks(xb, 128, 128)
    a = O.quant_error(xb, q, s, 128, 128, 128, 128)
    b = O.quant_error(xb, q, s, 128, 128, 1, 128)
    x = _bf16_val(xb)
    y32 = (O.e4m3_decode(q) * np.repeat(np.repeat(s, 128, 0), 128, 1).astype(np.float64))
    assert np.isclose(a[..., 2].sum(), np.sum(x * x), rtol=1e-12, atol=0)
    assert np.isclose(a[..., 1].sum(), b[..., 1].sum(), rtol=1e-12, atol=0)
    assert a[..., 0].max() == b[..., 0].max()
    assert a[..., 0].max() <= np.abs(x - y32).max() * (1 + 2.0 ** -20)


def test_kv_is_one_group_and_amax_matches_numpy():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((2, 64, 8, 128)) * np.exp(0.5 * rng.standard_normal((8, 128)))).astype(np.float32)
    xb = _bf16(x)
    q, scale, amax = O.kv_amax_quantize(xb)
    assert amax == np.abs(_f32(xb)).max()
    assert scale == np.float32(amax) / np.float32(448)
    q2, s2 = _library_quantize(xb.reshape(1, -1), 1, xb.size)
    assert (q.reshape(1, -1) == q2).all() and s2[0, 0] == scale
    assert (O.quantize_with_scale(xb, scale) == q).all()


# -------------------------------------------------------------------- GEMMs

def _rand_q(rng, m, k, scale_range=(1e-3, 1e-1)):
    xq = rng.integers(0, 256, (m, k), dtype=np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    return xq


def _dequant_numpy(q, s, br, bc):
    """Dequantize with the library codec and numpy broadcasting."""
    vals = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    full = np.repeat(np.repeat(s.astype(np.float64), br, 0), bc, 1)[:q.shape[0], :q.shape[1]]
    return vals * full


@pytest.mark.parametrize("m,n,k", [(1, 16, 128), (3, 130, 256), (64, 256, 512), (17, 48, 384)])
def test_gemm_matches_fp64_brute_force(m, n, k):
    rng = np.random.default_rng(m * 1000 + n)
    xq, wq = _rand_q(rng, m, k), _rand_q(rng, n, k)
    xs = rng.uniform(1e-3, 1e-1, (m, k // 128)).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-2, (-(-n // 128), k // 128)).astype(np.float32)
    y, absref = O.block_gemm(xq, xs, wq, ws)
    a = _dequant_numpy(xq, xs, 1, 128)
    b = _dequant_numpy(wq, ws, 128, 128)
    yb = a @ b.T
    ab = np.abs(a) @ np.abs(b).T
    assert np.allclose(absref, ab, rtol=1e-12, atol=0)
    assert (np.abs(y - yb) <= 1e-12 * ab + 1e-300).all()


def test_gemm_integer_case_is_exact():
    rng = np.random.default_rng(8)
    ints = np.arange(-8, 9)
    codes = O.e4m3_encode(ints.astype(np.float32))
    xi = rng.integers(0, len(ints), (9, 256))
    wi = rng.integers(0, len(ints), (20, 256))
    y, _ = O.block_gemm(codes[xi], np.ones((9, 2), np.float32), codes[wi], np.ones((1, 2), np.float32))
    exact = ints[xi].astype(np.int64) @ ints[wi].astype(np.int64).T
    assert (y == exact).all()


def test_gemm_single_slab_and_power_of_two_scaling():
    rng = np.random.default_rng(9)
    xq, wq = _rand_q(rng, 4, 128), _rand_q(rng, 8, 128)
    xs = np.array([[0.5], [0.25], [3.0], [1.0]], np.float32)
    ws = np.array([[0.125]], np.float32)
    y, _ = O.block_gemm(xq, xs, wq, ws)
    dx = torch.from_numpy(xq).view(torch.float8_e4m3fn).double().numpy()
    dw = torch.from_numpy(wq).view(torch.float8_e4m3fn).double().numpy()
    assert (y == (dx @ dw.T) * xs.astype(np.float64) * 0.125).all()
    y2, _ = O.block_gemm(xq, xs, wq, ws * np.float32(8))
    assert (y2 == y * 8).all()


def test_gemm_sensitivity_to_plausible_mistakes():
    """A transposed scale grid or a dropped slab must move the result by far
    more than the tolerance the GPU is held to."""
    rng = np.random.default_rng(10)
    m, n, k = 8, 256, 384
    xq, wq = _rand_q(rng, m, k), _rand_q(rng, n, k)
    xs = rng.uniform(1e-3, 1e-1, (m, 3)).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-2, (2, 3)).astype(np.float32)
    y, absref = O.block_gemm(xq, xs, wq, ws)
    tol = 1e-3 * absref
    ws_wrong = ws[::-1].copy()
    yw, _ = O.block_gemm(xq, xs, wq, ws_wrong)
    assert (np.abs(yw - y) > tol).mean() > 0.5
    xs_drop = xs.copy()
    xs_drop[:, 1] = 0
    yd, _ = O.block_gemm(xq, xs_drop, wq, ws)
    assert (np.abs(yd - y) > tol).mean() > 0.5


def test_gemm_entries_and_f32_variant():
    rng = np.random.default_rng(11)
    m, n, k = 12, 160, 512
    xq, wq = _rand_q(rng, m, k), _rand_q(rng, n, k)
    xs = rng.uniform(1e-3, 1e-1, (m, 4)).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-2, (2, 4)).astype(np.float32)
    y, absref = O.block_gemm(xq, xs, wq, ws)
    ii = rng.integers(0, m, 50)
    jj = rng.integers(0, n, 50)
    ye, ae = O.block_gemm_entries(xq, xs, wq, ws, ii, jj)
    assert (ye == y[ii, jj]).all() and (ae == absref[ii, jj]).all()
    y32 = O.block_gemm_f32acc(xq, xs, wq, ws)
    assert (np.abs(y32 - y) <= 1e-5 * absref).all()


def test_grouped_gemm_reduces_to_dense():
    rng = np.random.default_rng(12)
    g, n, k, rows = 5, 144, 256, 40
    xq = _rand_q(rng, rows, k)
    xs = rng.uniform(1e-3, 1e-1, (rows, 2)).astype(np.float32)
    wq = np.stack([_rand_q(rng, n, k) for _ in range(g)])
    ws = rng.uniform(1e-4, 1e-2, (g, 2, 2)).astype(np.float32)
    off = np.array([0, 7, 7, 30, 61, 90], np.int32)  # includes an empty group
    row_idx = rng.integers(0, rows, 90).astype(np.int32)
    y, a = O.grouped_gemm(xq, xs, row_idx, off, wq, ws)
    for e in range(g):
        r0, r1 = off[e], off[e + 1]
        yd, ad = O.block_gemm(xq[row_idx[r0:r1]], xs[row_idx[r0:r1]], wq[e], ws[e])
        assert (y[r0:r1] == yd).all() and (a[r0:r1] == ad).all()
    # one group with the identity gather is the dense GEMM
    y1, _ = O.grouped_gemm(xq, xs, None, np.array([0, rows], np.int32), wq[:1], ws[:1])
    yd, _ = O.block_gemm(xq, xs, wq[0], ws[0])
    assert (y1 == yd).all()


def test_bf16_rounding_matches_library_on_binary32_values():
    rng = np.random.default_rng(13)
    x = (rng.standard_normal(200000) * rng.choice([1e-30, 1e-3, 1, 1e4], 200000)).astype(np.float32)
    # include exact BF16 ties
    ties = ((rng.integers(0, 1 << 16, 1000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties[np.isfinite(ties)]])
    ours = O.bf16_from_f64(x.astype(np.float64))
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (ours == lib).all()
