/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the FP8 W8A8 hot path
 * computes.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this library; the product path never does.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * Sources (page title, then the section / table / equation):
 *   [FP8-RL]  "FP8-RL: A Practical and Stable Low-Precision Stack for LLM
 *             Reinforcement Learning" (dcwnkz.com write-up), section 1 "dynamic
 *             weight sync": E4M3, range [-448, 448], 128x128 weight blocks,
 *             dynamic activation quantization.
 *   [UFP8]    "Unified FP8: Moving Beyond Mixed Precision for Stable and
 *             Accelerated MoE RL" (papercache notes), quick-read section: the
 *             scale equation S = max|X| / V_max and the quantization equation
 *             Q(x) = round(x / S); section "FP8 scale choice": FP32 scales.
 *   [NeMo]    "NeMo RL FP8" (nvidia.csdn.net), Table 1 (weights [128,128],
 *             input activations [1,128], FP32 block scales) and Table 3
 *             (per-tensor FP32 scales for the stored KV cache).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - "round" is round-to-nearest, ties to even mantissa, onto the E4M3 grid,
 *     and magnitudes above 448 saturate to 448.
 *   - x / S is one IEEE binary32 division of the binary32 value of x by the
 *     binary32 scale S, and S = amax / 448 is one IEEE binary32 division.
 *   - An all-zero group gets S = 1.  Signed zero keeps its sign (-0 -> 0x80).
 *   - Edge blocks/groups that overhang the matrix use only in-bounds elements.
 *   - Scale grids are row-major: weights [ceil(N/128), ceil(K/128)],
 *     activations [M, ceil(K/128)].
 *   - The GEMM is Y = X W^T with W stored [N, K]; Y[i,j] is the sum over
 *     128-wide K slabs kb of xs[i,kb] * ws[j/128,kb] * sum_{k in kb} a*b.
 *
 * Build flags matter: -O2 -fno-fast-math -ffp-contract=off, so that every
 * binary32 '/' below is a single correctly rounded IEEE division and no
 * multiply-add is fused.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* BF16 and E4M3 value definitions                                           */
/* ------------------------------------------------------------------------ */

/* BF16 is the top half of a binary32 word, so widening is exact. */
ORACLE_EXPORT float oracle_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * E4M3 decode from the format definition ([UFP8] "FP8 data formats", which
 * refers to the OCP 8-bit floating point specification): 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal;
 * S.1111.111 is NaN and there is no infinity, so the largest finite
 * magnitude is 1.75 * 2^8 = 448 ([FP8-RL] section 1 gives the range).
 */
ORACLE_EXPORT double oracle_e4m3_decode(uint8_t code) {
    int s = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7); /* 0.m * 2^(1-bias) */
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7); /* 1.m * 2^(e-bias) */
    return s ? -mag : mag;
}

/*
 * Encoder A: nearest point of the E4M3 grid, found by search, ties to the
 * code with the even mantissa (the code's last bit), magnitudes >= 448
 * saturated to 448.  Slow and plain on purpose.
 *
 * Exactness: for |v| >= 2^-10 the distances below are multiples of 2^-33 of
 * size < 2^9, so double holds them exactly; for |v| < 2^-10 code 0 wins with
 * room to spare, so rounding of the distances cannot change the answer.
 */
ORACLE_EXPORT uint8_t oracle_e4m3_encode(float v) {
    uint8_t sign;
    double a;
    int lo, hi;
    if (v != v) return 0x7F; /* NaN: outside the contract */
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    /* codes 0..126 are the non-negative finite values in increasing order */
    lo = 0;
    hi = 126;
    while (hi - lo > 1) { /* invariant: decode(lo) <= a < decode(hi) */
        int mid = (lo + hi) / 2;
        if (oracle_e4m3_decode((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    {
        double dlo = a - oracle_e4m3_decode((uint8_t)lo);
        double dhi = oracle_e4m3_decode((uint8_t)hi) - a;
        int c;
        if (dlo < dhi)
            c = lo;
        else if (dhi < dlo)
            c = hi;
        else
            c = (lo % 2 == 0) ? lo : hi;
        return (uint8_t)(sign | c);
    }
}

/*
 * Encoder B: the same rounding done on the binary32 bit fields.  Written
 * differently from encoder A so that an exhaustive sweep of one against the
 * other catches a slip in either; the tests pin A and B to each other and to
 * torch's float8_e4m3fn conversion.
 */
ORACLE_EXPORT uint8_t oracle_e4m3_encode_bits(float v) {
    uint32_t u, a, sig, k, rest, half;
    int e, shift;
    uint8_t sign;
    memcpy(&u, &v, sizeof u);
    sign = (uint8_t)((u >> 24) & 0x80);
    a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return 0x7F;               /* NaN */
    if (a >= 0x43E00000u) return (uint8_t)(sign | 0x7E); /* |v| >= 448 */
    e = (int)(a >> 23) - 127;
    if (e < -10) return sign; /* |v| < 2^-10: nearer to 0 than to 2^-9 */
    sig = (a & 0x7FFFFFu) | 0x800000u; /* |v| = sig * 2^(e-23) */
    if (e >= -6) {
        /* normal E4M3: keep 3 of the 23 stored mantissa bits */
        uint32_t keep = (a & 0x7FFFFFu) >> 20;
        int be = e + 7;
        rest = a & 0xFFFFFu;
        half = 0x80000u;
        if (rest > half || (rest == half && (keep & 1u))) keep += 1;
        if (keep == 8) {
            keep = 0;
            be += 1;
        }
        return (uint8_t)(sign | (uint32_t)(be << 3) | keep);
    }
    /* subnormal E4M3: |v| / 2^-9 = sig * 2^(e+9-23), rounded to an integer */
    shift = 14 - e; /* 21..24 for e = -7..-10 */
    k = sig >> shift;
    rest = sig & ((1u << shift) - 1u);
    half = 1u << (shift - 1);
    if (rest > half || (rest == half && (k & 1u))) k += 1;
    /* k == 8 is 2^-6, the smallest normal, whose code is also 8 */
    return (uint8_t)(sign | k);
}

/* Exhaustive helper: compares encoders A and B on the binary32 bit patterns
 * [start, start+count), skipping NaNs.  Returns the number of mismatches and
 * stores the first mismatching pattern in *first. */
ORACLE_EXPORT int64_t oracle_e4m3_cross_check(uint32_t start, uint64_t count,
                                               uint32_t *first) {
    int64_t bad = 0;
    uint64_t i;
    for (i = 0; i < count; ++i) {
        uint32_t b = (uint32_t)(start + i);
        float v;
        if ((b & 0x7FFFFFFFu) > 0x7F800000u) continue;
        memcpy(&v, &b, sizeof v);
        if (oracle_e4m3_encode(v) != oracle_e4m3_encode_bits(v)) {
            if (bad == 0 && first) *first = b;
            ++bad;
        }
    }
    return bad;
}

/* Fills codes[i] = encoder B applied to the binary32 pattern start+i.  Used
 * to state the expected hardware conversion result over all patterns. */
ORACLE_EXPORT void oracle_e4m3_encode_patterns(uint32_t start, uint64_t count,
                                               uint8_t *codes) {
    uint64_t i;
    for (i = 0; i < count; ++i) {
        uint32_t b = (uint32_t)(start + i);
        float v;
        memcpy(&v, &b, sizeof v);
        codes[i] = oracle_e4m3_encode_bits(v);
    }
}

ORACLE_EXPORT void oracle_e4m3_encode_array(const float *x, int64_t n,
                                            uint8_t *q) {
    int64_t i;
    for (i = 0; i < n; ++i) q[i] = oracle_e4m3_encode(x[i]);
}

ORACLE_EXPORT void oracle_e4m3_decode_array(const uint8_t *q, int64_t n,
                                            double *y) {
    int64_t i;
    for (i = 0; i < n; ++i) y[i] = oracle_e4m3_decode(q[i]);
}

/* ------------------------------------------------------------------------ */
/* Quantization ([UFP8] scale and quantization equations)                    */
/* ------------------------------------------------------------------------ */

/* S = max|X| / V_max with V_max = 448, one binary32 division; S := 1 when
 * the group is all zeros (the pages are silent; this keeps x/S defined). */
ORACLE_EXPORT float oracle_scale_from_amax(float amax) {
    if (amax == 0.0f) return 1.0f;
    return amax / 448.0f;
}

/* Q(x) = round(x / S): binary32 division, then E4M3 rounding with
 * saturation. */
/* Power-of-two scale ([NeMo] blog, recipe variants: "power-of-2 scaling
 * factor"): the smallest power of two S with 448 * S >= amax, found by
 * walking the exponent with exact comparisons (448 * 2^e is exact in
 * binary32 over the whole range used); S = 1 for an all-zero group. */
ORACLE_EXPORT float oracle_scale_pow2_from_amax(float amax) {
    int e = 0;
    if (amax == 0.0f) return 1.0f;
    while (448.0f * ldexpf(1.0f, e) < amax) ++e;
    while (448.0f * ldexpf(1.0f, e - 1) >= amax) --e;
    return ldexpf(1.0f, e);
}

ORACLE_EXPORT uint8_t oracle_quantize_value(float x, float s) {
    float t = x / s;
    return oracle_e4m3_encode(t);
}

/*
 * Generic block quantizer.  x is a row-major [rows, cols] BF16 matrix.  It is
 * tiled into br x bc blocks (edge blocks overhang and use only in-bounds
 * elements); each block gets one FP32 scale from its own amax, stored
 * row-major in s[ceil(rows/br), ceil(cols/bc)], and every element is coded
 * with its block's scale into q[rows, cols].
 *   weights:      br = bc = 128        ([FP8-RL] sec. 1; [NeMo] Table 1)
 *   activations:  br = 1,  bc = 128    ([NeMo] Table 1; [UFP8] per-token)
 *   KV cache:     rows = 1, br = 1, bc = cols = numel  ([NeMo] Table 3)
 */
/* pow2 != 0: power-of-two scales (oracle_scale_pow2_from_amax). */
ORACLE_EXPORT int oracle_quantize_blocks_mode(const uint16_t *x, int64_t rows,
                                              int64_t cols, int64_t br, int64_t bc,
                                              int pow2, uint8_t *q, float *s) {
    int64_t nbr, nbc, bi, bj, r, c;
    if (rows < 0 || cols < 0 || br <= 0 || bc <= 0) return -1;
    nbr = (rows + br - 1) / br;
    nbc = (cols + bc - 1) / bc;
    for (bi = 0; bi < nbr; ++bi) {
        for (bj = 0; bj < nbc; ++bj) {
            int64_t r0 = bi * br, r1 = r0 + br < rows ? r0 + br : rows;
            int64_t c0 = bj * bc, c1 = c0 + bc < cols ? c0 + bc : cols;
            float amax = 0.0f, scale;
            for (r = r0; r < r1; ++r)
                for (c = c0; c < c1; ++c) {
                    float a = fabsf(oracle_bf16_to_f32(x[r * cols + c]));
                    if (a > amax) amax = a;
                }
            scale = pow2 ? oracle_scale_pow2_from_amax(amax) : oracle_scale_from_amax(amax);
            s[bi * nbc + bj] = scale;
            for (r = r0; r < r1; ++r)
                for (c = c0; c < c1; ++c)
                    q[r * cols + c] =
                        oracle_quantize_value(oracle_bf16_to_f32(x[r * cols + c]), scale);
        }
    }
    return 0;
}

ORACLE_EXPORT int oracle_quantize_blocks(const uint16_t *x, int64_t rows,
                                         int64_t cols, int64_t br, int64_t bc,
                                         uint8_t *q, float *s) {
    return oracle_quantize_blocks_mode(x, rows, cols, br, bc, 0, q, s);
}

/* max |x| over a BF16 array (the per-tensor KV amax). */
ORACLE_EXPORT float oracle_amax_bf16(const uint16_t *x, int64_t n) {
    float amax = 0.0f;
    int64_t i;
    for (i = 0; i < n; ++i) {
        float a = fabsf(oracle_bf16_to_f32(x[i]));
        if (a > amax) amax = a;
    }
    return amax;
}

/* Quantize with a given scale (the KV "quantize only" mode, where the scale
 * from an earlier recalibration is reused). */
ORACLE_EXPORT void oracle_quantize_with_scale(const uint16_t *x, int64_t n,
                                              float scale, uint8_t *q) {
    int64_t i;
    for (i = 0; i < n; ++i)
        q[i] = oracle_quantize_value(oracle_bf16_to_f32(x[i]), scale);
}

/* ------------------------------------------------------------------------ */
/* Blockwise-scaled FP8 GEMM ([NeMo] Table 1 granularities)                   */
/* ------------------------------------------------------------------------ */

/*
 * One output element of Y = X W^T:
 *   Y[i,j] = sum_kb xs[i,kb] * ws[j/128,kb] * sum_{k in slab kb} dec(xq[i,k]) dec(wq[j,k])
 * Each product of two E4M3 values is exact in double and a 128-term slab sum
 * of them is exact too (multiples of 2^-18 below 2^25), so the only rounding
 * is in the final scale-and-sum, done in double.  *absref receives
 * sum_k |dec(a) xs * dec(b) ws|, the scale the error tolerance is stated in.
 */
static void gemm_entry(const uint8_t *xrow, const float *xsrow,
                       const uint8_t *wrow, const float *wsrow, int64_t k,
                       double *y, double *absref) {
    int64_t nkb = (k + 127) / 128, kb, kk;
    double acc = 0.0, accabs = 0.0;
    for (kb = 0; kb < nkb; ++kb) {
        int64_t k0 = kb * 128, k1 = k0 + 128 < k ? k0 + 128 : k;
        double dot = 0.0, dotabs = 0.0;
        double sab = (double)xsrow[kb] * (double)wsrow[kb];
        for (kk = k0; kk < k1; ++kk) {
            double p = oracle_e4m3_decode(xrow[kk]) * oracle_e4m3_decode(wrow[kk]);
            dot += p;
            dotabs += fabs(p);
        }
        acc += dot * sab;
        accabs += dotabs * fabs(sab);
    }
    *y = acc;
    *absref = accabs;
}

/* Dense GEMM over all (i, j): xq [m,k], xs [m,ceil(k/128)], wq [n,k],
 * ws [ceil(n/128), ceil(k/128)], y and absref [m,n] in double. */
ORACLE_EXPORT int oracle_block_gemm(const uint8_t *xq, const float *xs,
                                    const uint8_t *wq, const float *ws,
                                    int64_t m, int64_t n, int64_t k, double *y,
                                    double *absref) {
    int64_t nkb = (k + 127) / 128, i, j;
    if (m < 0 || n < 0 || k < 0) return -1;
    for (i = 0; i < m; ++i)
        for (j = 0; j < n; ++j)
            gemm_entry(xq + i * k, xs + i * nkb, wq + j * k, ws + (j / 128) * nkb,
                       k, &y[i * n + j], &absref[i * n + j]);
    return 0;
}

/* The same definition on a list of (i, j) entries, for sampled parity at
 * sizes where the full product would take the CPU too long. */
ORACLE_EXPORT int oracle_block_gemm_entries(const uint8_t *xq, const float *xs,
                                            const uint8_t *wq, const float *ws,
                                            int64_t k, const int64_t *ii,
                                            const int64_t *jj, int64_t count,
                                            double *y, double *absref) {
    int64_t nkb = (k + 127) / 128, t;
    for (t = 0; t < count; ++t)
        gemm_entry(xq + ii[t] * k, xs + ii[t] * nkb, wq + jj[t] * k,
                   ws + (jj[t] / 128) * nkb, k, &y[t], &absref[t]);
    return 0;
}

/*
 * Diagnostic variant with binary32 arithmetic in the order a blockwise FP8
 * kernel would use: each slab's dot accumulated in FP32, then
 * acc += dot * (xs * ws) in FP32.  Not the reference result; the tests use it
 * only to show how far an FP32-accumulating kernel may sit from the exact one.
 */
ORACLE_EXPORT int oracle_block_gemm_f32acc(const uint8_t *xq, const float *xs,
                                           const uint8_t *wq, const float *ws,
                                           int64_t m, int64_t n, int64_t k,
                                           float *y) {
    int64_t nkb = (k + 127) / 128, i, j, kb, kk;
    for (i = 0; i < m; ++i)
        for (j = 0; j < n; ++j) {
            float acc = 0.0f;
            for (kb = 0; kb < nkb; ++kb) {
                int64_t k0 = kb * 128, k1 = k0 + 128 < k ? k0 + 128 : k;
                float dot = 0.0f, sab;
                for (kk = k0; kk < k1; ++kk)
                    dot += (float)(oracle_e4m3_decode(xq[i * k + kk]) *
                                   oracle_e4m3_decode(wq[j * k + kk]));
                sab = xs[i * nkb + kb] * ws[(j / 128) * nkb + kb];
                acc += dot * sab;
            }
            y[i * n + j] = acc;
        }
    return 0;
}

/*
 * Grouped (MoE) GEMM: rows [off[e], off[e+1]) of the output belong to expert
 * e; output row r reads activation row src = row_idx ? row_idx[r] : r and
 * expert e's weights wq + e*n*k with scale grid ws + e*ceil(n/128)*ceil(k/128).
 * Each row is the dense definition above.  y and absref are [off[g], n].
 */
ORACLE_EXPORT int oracle_grouped_gemm(const uint8_t *xq, const float *xs,
                                      int64_t rows_x, const int32_t *row_idx,
                                      const int32_t *group_offsets, int32_t g,
                                      const uint8_t *wq, const float *ws,
                                      int64_t n, int64_t k, double *y,
                                      double *absref) {
    int64_t nkb = (k + 127) / 128, nnb = (n + 127) / 128, r, j;
    int32_t e;
    for (e = 0; e < g; ++e) {
        const uint8_t *we = wq + (int64_t)e * n * k;
        const float *wse = ws + (int64_t)e * nnb * nkb;
        for (r = group_offsets[e]; r < group_offsets[e + 1]; ++r) {
            int64_t src = row_idx ? row_idx[r] : r;
            if (src < 0 || src >= rows_x) return -1;
            for (j = 0; j < n; ++j)
                gemm_entry(xq + src * k, xs + src * nkb, we + j * k,
                           wse + (j / 128) * nkb, k, &y[r * n + j],
                           &absref[r * n + j]);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequantization (fake quant) and the quantization-error report             */
/* ------------------------------------------------------------------------ */

/* The inverse the pages pair with Q in their error analysis ([UFP8] "fake
 * quant" vs "real quant" experiments): x_hat = dec(q) * S as one binary32
 * multiply.  dec(q) is exact in binary32. */
ORACLE_EXPORT float oracle_dequant_value(uint8_t q, float s) {
    float d = (float)oracle_e4m3_decode(q);
    return d * s;
}

uint16_t oracle_bf16_from_f64(double y);

/* Dequantize a block-scaled matrix to BF16: y = BF16_RN(x_hat), scale of
 * element (r, c) at s[(r / br) * ceil(cols / bc) + c / bc]. */
ORACLE_EXPORT int oracle_dequantize_blocks(const uint8_t *q, const float *s, int64_t rows,
                                           int64_t cols, int64_t br, int64_t bc,
                                           uint16_t *y) {
    int64_t r, c, nbc;
    if (rows < 0 || cols < 0 || br <= 0 || bc <= 0) return -1;
    nbc = (cols + bc - 1) / bc;
    for (r = 0; r < rows; ++r)
        for (c = 0; c < cols; ++c)
            y[r * cols + c] = oracle_bf16_from_f64(
                (double)oracle_dequant_value(q[r * cols + c], s[(r / br) * nbc + c / bc]));
    return 0;
}

/* Quantization-error report over report blocks of rbr x rbc elements (the
 * quantization blocks, sbr x sbc, are given separately): per report block,
 * stats[3*b + 0] = max |x - x_hat|, stats[3*b + 1] = sum (x - x_hat)^2,
 * stats[3*b + 2] = sum x^2, all in FP64, elements taken in row-major order
 * inside the block; x_hat is the binary32 dequantized value. */
ORACLE_EXPORT int oracle_quant_error(const uint16_t *x, const uint8_t *q, const float *s,
                                     int64_t rows, int64_t cols, int64_t sbr, int64_t sbc,
                                     int64_t rbr, int64_t rbc, double *stats) {
    int64_t nsbc, nrbr, nrbc, br, bc, r, c;
    if (rows < 0 || cols < 0 || sbr <= 0 || sbc <= 0 || rbr <= 0 || rbc <= 0) return -1;
    nsbc = (cols + sbc - 1) / sbc;
    nrbr = (rows + rbr - 1) / rbr;
    nrbc = (cols + rbc - 1) / rbc;
    for (br = 0; br < nrbr; ++br)
        for (bc = 0; bc < nrbc; ++bc) {
            double mx = 0.0, se = 0.0, sx = 0.0;
            for (r = br * rbr; r < rows && r < (br + 1) * rbr; ++r)
                for (c = bc * rbc; c < cols && c < (bc + 1) * rbc; ++c) {
                    double xv = (double)oracle_bf16_to_f32(x[r * cols + c]);
                    double xh = (double)oracle_dequant_value(q[r * cols + c],
                                                             s[(r / sbr) * nsbc + c / sbc]);
                    double e = xv - xh;
                    if (fabs(e) > mx) mx = fabs(e);
                    se += e * e;
                    sx += xv * xv;
                }
            stats[3 * (br * nrbc + bc) + 0] = mx;
            stats[3 * (br * nrbc + bc) + 1] = se;
            stats[3 * (br * nrbc + bc) + 2] = sx;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decode attention over the FP8 KV cache                                    */
/* ------------------------------------------------------------------------ */

/* [NeMo] Table 3 and the FP8 KV-cache section: Q, K and V carry one FP32
 * scale each (per tensor); [FP8-RL] section 4: attention reads the FP8 KV
 * cache.  One query token per sequence b and query head h, grouped-query
 * attention (query head h reads KV head h / (hq / hkv)):
 *   score_t = softmax_scale * sq * sk * sum_d dec(q[b,h,d]) dec(k[b,t,kh,d])
 *   p_t     = exp(score_t - max) / sum_u exp(score_u - max),   t < len_b
 *   out_d   = sv * sum_t p_t dec(v[b,t,kh,d])
 * all in FP64; absout_d = sv * sum_t p_t |dec(v)| bounds the rounding.  An
 * empty sequence gives out = 0. */
ORACLE_EXPORT int oracle_decode_attention(const uint8_t *q, float sq, const uint8_t *k, float sk,
                                          const uint8_t *v, float sv, const int32_t *lens,
                                          int64_t batch, int64_t smax, int64_t hq, int64_t hkv,
                                          int64_t d, double softmax_scale, double *out,
                                          double *absout) {
    int64_t b, h, t, i;
    double dec[256];
    if (batch < 0 || smax < 0 || hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv) return -1;
    for (i = 0; i < 256; ++i) dec[i] = oracle_e4m3_decode((uint8_t)i); /* the codec above, tabulated */
    for (b = 0; b < batch; ++b) {
        int64_t len = lens[b];
        if (len < 0 || len > smax) return -2;
        for (h = 0; h < hq; ++h) {
            int64_t kh = h / (hq / hkv);
            const uint8_t *qv = q + (b * hq + h) * d;
            double *o = out + (b * hq + h) * d;
            double *ao = absout + (b * hq + h) * d;
            double mx = -HUGE_VAL, den = 0.0;
            for (i = 0; i < d; ++i) o[i] = ao[i] = 0.0;
            if (len == 0) continue;
            for (t = 0; t < len; ++t) {
                const uint8_t *kv = k + ((b * smax + t) * hkv + kh) * d;
                double sc = 0.0;
                for (i = 0; i < d; ++i) sc += dec[qv[i]] * dec[kv[i]];
                sc *= softmax_scale * (double)sq * (double)sk;
                if (sc > mx) mx = sc;
            }
            for (t = 0; t < len; ++t) {
                const uint8_t *kv = k + ((b * smax + t) * hkv + kh) * d;
                const uint8_t *vv = v + ((b * smax + t) * hkv + kh) * d;
                double sc = 0.0, pt;
                for (i = 0; i < d; ++i) sc += dec[qv[i]] * dec[kv[i]];
                sc *= softmax_scale * (double)sq * (double)sk;
                pt = exp(sc - mx);
                den += pt;
                for (i = 0; i < d; ++i) {
                    double x = dec[vv[i]];
                    o[i] += pt * x;
                    ao[i] += pt * fabs(x);
                }
            }
            for (i = 0; i < d; ++i) {
                o[i] = o[i] / den * (double)sv;
                ao[i] = ao[i] / den * fabs((double)sv);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Prefill (causal) attention over FP8 Q, K and V                            */
/* ------------------------------------------------------------------------ */

/* [NeMo] Table 3: Q, K and V carry one FP32 scale each (per tensor); the
 * prompt's tokens attend causally: query token i of sequence b, query head h,
 * reads the keys and values of tokens 0..i of the same sequence, KV head
 * h / (hq / hkv).  q [batch, seq, hq, d], k and v [batch, seq, hkv, d]:
 *   score_j = softmax_scale * sq * sk * sum_d dec(q[b,i,h,d]) dec(k[b,j,kh,d])
 *   p_j     = exp(score_j - max) / sum_{u <= i} exp(score_u - max),  j <= i
 *   out_d   = sv * sum_{j <= i} p_j dec(v[b,j,kh,d])
 * all in FP64; absout_d = sv * sum_j p_j |dec(v)| bounds the rounding.  The
 * scores of a row are formed once and kept (seq <= 1 << 20). */
ORACLE_EXPORT int oracle_prefill_attention(const uint8_t *q, float sq, const uint8_t *k, float sk,
                                           const uint8_t *v, float sv, int64_t batch, int64_t seq,
                                           int64_t hq, int64_t hkv, int64_t d,
                                           double softmax_scale, double *out, double *absout) {
    int64_t b, h, i, j, e;
    double dec[256];
    double *sc;
    if (batch < 0 || seq < 0 || seq > (1 << 20) || hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv)
        return -1;
    for (e = 0; e < 256; ++e) dec[e] = oracle_e4m3_decode((uint8_t)e);
    sc = (double *)malloc(sizeof(double) * (size_t)(seq > 0 ? seq : 1));
    if (!sc) return -3;
    for (b = 0; b < batch; ++b)
        for (i = 0; i < seq; ++i)
            for (h = 0; h < hq; ++h) {
                const int64_t kh = h / (hq / hkv);
                const uint8_t *qv = q + ((b * seq + i) * hq + h) * d;
                double *o = out + ((b * seq + i) * hq + h) * d;
                double *ao = absout + ((b * seq + i) * hq + h) * d;
                double mx = -HUGE_VAL, den = 0.0;
                for (e = 0; e < d; ++e) o[e] = ao[e] = 0.0;
                for (j = 0; j <= i; ++j) {
                    const uint8_t *kv = k + ((b * seq + j) * hkv + kh) * d;
                    double s = 0.0;
                    for (e = 0; e < d; ++e) s += dec[qv[e]] * dec[kv[e]];
                    s *= softmax_scale * (double)sq * (double)sk;
                    sc[j] = s;
                    if (s > mx) mx = s;
                }
                for (j = 0; j <= i; ++j) {
                    const uint8_t *vv = v + ((b * seq + j) * hkv + kh) * d;
                    const double pj = exp(sc[j] - mx);
                    den += pj;
                    for (e = 0; e < d; ++e) {
                        const double x = dec[vv[e]];
                        o[e] += pj * x;
                        ao[e] += pj * fabs(x);
                    }
                }
                for (e = 0; e < d; ++e) {
                    o[e] = o[e] / den * (double)sv;
                    ao[e] = ao[e] / den * fabs((double)sv);
                }
            }
    free(sc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Output rounding                                                            */
/* ------------------------------------------------------------------------ */

/* Round a double to the nearest BF16 (8 significant bits), ties to even, in
 * one step.  Finite inputs whose magnitude is below 2^-133 or above the BF16
 * range are outside what the tests produce; they go to 0 / infinity. */
ORACLE_EXPORT uint16_t oracle_bf16_from_f64(double y) {
    int e;
    double f, scaled, ip, frac;
    uint32_t u, mag;
    float out;
    if (y != y) return 0x7FC0;
    if (y == 0.0) return signbit(y) ? 0x8000 : 0x0000;
    f = frexp(fabs(y), &e); /* |y| = f * 2^e, f in [0.5, 1) */
    if (e - 1 < -126) {
        /* BF16 subnormal: quantum 2^-133 */
        scaled = ldexp(fabs(y), 133);
    } else {
        scaled = ldexp(f, 8); /* [128, 256): 8 significant bits in the integer part */
    }
    frac = modf(scaled, &ip);
    if (frac > 0.5 || (frac == 0.5 && fmod(ip, 2.0) != 0.0)) ip += 1.0;
    if (e - 1 < -126)
        out = (float)ldexp(ip, -133);
    else
        out = (float)ldexp(ip, e - 8);
    memcpy(&u, &out, sizeof u);
    mag = u >> 16;
    return (uint16_t)(signbit(y) ? (mag | 0x8000) : mag);
}

ORACLE_EXPORT void oracle_bf16_from_f64_array(const double *y, int64_t n,
                                              uint16_t *out) {
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = oracle_bf16_from_f64(y[i]);
}
