/*
 * Grouped INT2 encoding of the rotated latent, plain C (oracle, test
 * infrastructure only; shares nothing with the CUDA path).
 *
 * Source: "MLA model support (GLM-5.1 / DeepSeek-style)" (OSCAR issue #10),
 * maintainer reply, "How the rotation adapts to the latent": the cache holds
 * the rotated + quantised latent, low-variance directions share INT2 groups,
 * clip thresholds are fit on the rotated latent, attention reads the
 * dequantised latent.
 *
 * Readings adopted where the page gives no formula (the integer codes are
 * decided here, so the operation order below is part of the definition):
 *   rotation   y_j = fmaf chain over k = 0..r-1 ascending of c_k * R[k][j],
 *              starting from +0.0f, fp32 (R row-major [r][r], y = c . R).
 *   clip       yc = min(max(y, -T_g), T_g), group g = j / gs.
 *   range      lo = min_j yc, hi = max_j yc over the group.
 *   scale/zero s = fp16_rne((hi - lo) / 3.0f), z = fp16_rne(lo), both then
 *              widened back to fp32.
 *   code       s == 0 -> 0; else clamp(rint_even((yc - z) / s), 0, 3) with
 *              fp32 subtraction and IEEE division, no contraction.
 *   packing    element j of a group -> byte j/4 of the group's gs/4 bytes,
 *              bits 2*(j%4) .. 2*(j%4)+1 (least significant first); group g
 *              occupies bytes g*gs/4 .. of the token's r/4-byte code row.
 *   dequant    c^_j = fmaf(code, s, z).
 *
 * Built with -ffp-contract=off so no other multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint16_t f32_to_f16_bits(float x) {
    _Float16 h = (_Float16)x;          /* IEEE round-to-nearest-even */
    uint16_t b;
    memcpy(&b, &h, sizeof b);
    return b;
}

static float f16_bits_to_f32(uint16_t b) {
    _Float16 h;
    memcpy(&h, &b, sizeof h);
    return (float)h;
}

/* y[n][r] = c[n][r] . R[r][r], fp32 fused-multiply-add chain, ascending k. */
void oracle_rotate_chain(const float *c, const float *R, int64_t n, int r, float *y) {
    /* Each output keeps its own chain y_j <- fmaf(c_k, R[k][j], y_j) for
     * k = 0, 1, ..., r-1; the loops visit k outermost only so that R is read
     * row by row. */
    for (int64_t t = 0; t < n; ++t) {
        const float *ct = c + t * r;
        float *yt = y + t * r;
        for (int j = 0; j < r; ++j) yt[j] = 0.0f;
        for (int k = 0; k < r; ++k) {
            const float *Rk = R + (int64_t)k * r;
            for (int j = 0; j < r; ++j) yt[j] = fmaf(ct[k], Rk[j], yt[j]);
        }
    }
}

/* Encode already-rotated rows y[n][r]. codes[n][r/4] (u8), sz[n][r/gs][2]
 * (fp16 bit patterns: scale then zero). */
void oracle_int2_encode(const float *y, const float *T, int64_t n, int r, int gs,
                        uint8_t *codes, uint16_t *sz) {
    const int ng = r / gs;
    for (int64_t t = 0; t < n; ++t) {
        const float *yt = y + t * r;
        uint8_t *ct = codes + t * (r / 4);
        memset(ct, 0, (size_t)(r / 4));
        for (int g = 0; g < ng; ++g) {
            const float thr = T[g];
            float lo = INFINITY, hi = -INFINITY;
            for (int j = 0; j < gs; ++j) {
                float v = fminf(fmaxf(yt[g * gs + j], -thr), thr);
                lo = fminf(lo, v);
                hi = fmaxf(hi, v);
            }
            const uint16_t sb = f32_to_f16_bits((hi - lo) / 3.0f);
            const uint16_t zb = f32_to_f16_bits(lo);
            sz[(t * ng + g) * 2 + 0] = sb;
            sz[(t * ng + g) * 2 + 1] = zb;
            const float s = f16_bits_to_f32(sb), z = f16_bits_to_f32(zb);
            for (int j = 0; j < gs; ++j) {
                float v = fminf(fmaxf(yt[g * gs + j], -thr), thr);
                int code = 0;
                if (s != 0.0f) {
                    float qv = rintf((v - z) / s);
                    code = qv < 0.0f ? 0 : (qv > 3.0f ? 3 : (int)qv);
                }
                const int e = g * gs + j;
                ct[e / 4] |= (uint8_t)(code << (2 * (e % 4)));
            }
        }
    }
}

/* c^[n][r] from codes and fp16 scale/zero. */
void oracle_int2_decode(const uint8_t *codes, const uint16_t *sz, int64_t n, int r, int gs,
                        float *out) {
    const int ng = r / gs;
    for (int64_t t = 0; t < n; ++t) {
        for (int e = 0; e < r; ++e) {
            const int g = e / gs;
            const int code = (codes[t * (r / 4) + e / 4] >> (2 * (e % 4))) & 3;
            const float s = f16_bits_to_f32(sz[(t * ng + g) * 2 + 0]);
            const float z = f16_bits_to_f32(sz[(t * ng + g) * 2 + 1]);
            out[t * r + e] = fmaf((float)code, s, z);
        }
    }
}
