/*
 * oracle.c -- plain fp64 CPU oracle for hybrid-SWA attention with sinks.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  It shares no
 * code, header, table or constant generator with the CUDA path.
 *
 * What it computes is the plain definition of one attention layer of
 * MiMo-V2-style hybrid attention, written out with no ring, no pages, no
 * tiles and no blocking: keys are addressed by their token position.
 *
 *  - partial rotate-half RoPE on dims 0..63 of every 192-wide q/k head,
 *    inv_freq_i = theta^(-2i/64), angle = position * inv_freq_i, all in fp64
 *    (colibri "MiMo-V2.6", section "What the engine implements";
 *    gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", section "The RoPE fix for
 *    large positions": the cos/sin are computed in float64 on the CPU);
 *  - v' = v * value_scale (colibri, "What the engine implements": values are
 *    multiplied by attention_value_scale before attention);
 *  - s_j = (q'.k'_j) * softmax_scale over the key set J(p): {0..p} for a
 *    full-attention layer, {p-W+1..p} (W = 128, "exactly the last 128
 *    positions", gaudi-cookbook "What was built") for a windowed layer;
 *  - o = sum_j e^{s_j-m} v'_j / Z with Z = sum_j e^{s_j-m}, plus e^{sink-m}
 *    on windowed layers only: the sink "joins the softmax denominator and
 *    nothing else" (colibri, "What the engine implements").  m is the max of
 *    the logits and the sink; it cancels and only keeps exp() in range.
 *  - GQA: q head h reads kv head h / (Hq/Hkv).
 *
 * Inputs are the raw bf16 bit patterns, widened exactly to double.  Nothing
 * is rounded on the way; the result is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_DQK 192
#define ORC_DV 128
#define ORC_DROT 64
#define ORC_HALF 32

/* bf16 bits -> double, exact. */
static double orc_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), returning its bits.
 * Used only by the storage-faithful checks of the KV write. */
uint16_t orc_round_bf16(double x) {
    if (isnan(x)) return 0x7fc0;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    double a = fabs(x);
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int ulp_exp = (e - 1) - 7;    /* 7 fraction bits below the leading one */
    if (ulp_exp < -133) ulp_exp = -133;   /* bf16 subnormal spacing */
    double r = nearbyint(ldexp(a, -ulp_exp));   /* ties-to-even */
    double y = ldexp(r, ulp_exp);
    float f = (float)y;           /* exact: y has at most 8 significant bits */
    if (y > 3.3895313892515355e38) f = INFINITY;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t bits = (uint16_t)(u >> 16);
    if (signbit(x)) bits |= 0x8000;
    return bits;
}

/* cos/sin of every rotary frequency at one position, fp64.
 * cs[2i] = cos(pos * theta^(-2i/64)), cs[2i+1] = sin(...). */
void orc_rope_cos_sin(double theta, int64_t pos, double *cs) {
    for (int i = 0; i < ORC_HALF; ++i) {
        double inv_freq = pow(theta, -(2.0 * i) / (double)ORC_DROT);
        double ang = (double)pos * inv_freq;
        cs[2 * i] = cos(ang);
        cs[2 * i + 1] = sin(ang);
    }
}

/* Rotate-half RoPE of one 192-wide head (x given as doubles). */
static void orc_rope_apply(const double *x, const double *cs, double *out) {
    for (int i = 0; i < ORC_HALF; ++i) {
        double c = cs[2 * i], s = cs[2 * i + 1];
        double x1 = x[i], x2 = x[i + ORC_HALF];
        out[i] = x1 * c - x2 * s;
        out[i + ORC_HALF] = x2 * c + x1 * s;
    }
    for (int d = ORC_DROT; d < ORC_DQK; ++d) out[d] = x[d];
}

/* RoPE of raw bf16 heads: x [n][192] bf16 bits at positions pos[n] -> fp64. */
void orc_rope_heads(const uint16_t *x, const int64_t *pos, int64_t n, double theta, double *out) {
    double cs[2 * ORC_HALF], xd[ORC_DQK];
    for (int64_t r = 0; r < n; ++r) {
        orc_rope_cos_sin(theta, pos[r], cs);
        for (int d = 0; d < ORC_DQK; ++d) xd[d] = orc_bf16(x[r * ORC_DQK + d]);
        orc_rope_apply(xd, cs, out + r * ORC_DQK);
    }
}

/* The stored form of one KV write, rounded once to bf16: k' = RNE(rope(k)),
 * v' = RNE(v * value_scale).  k [n][hkv][192], v [n][hkv][128], pos [n]. */
void orc_kv_store_bf16(const uint16_t *k, const uint16_t *v, const int64_t *pos, int64_t n, int hkv,
                       double theta, double value_scale, uint16_t *k_out, uint16_t *v_out) {
    double cs[2 * ORC_HALF], xd[ORC_DQK], yd[ORC_DQK];
    for (int64_t r = 0; r < n; ++r) {
        orc_rope_cos_sin(theta, pos[r], cs);
        for (int h = 0; h < hkv; ++h) {
            const uint16_t *kr = k + (r * hkv + h) * ORC_DQK;
            for (int d = 0; d < ORC_DQK; ++d) xd[d] = orc_bf16(kr[d]);
            orc_rope_apply(xd, cs, yd);
            for (int d = 0; d < ORC_DQK; ++d) k_out[(r * hkv + h) * ORC_DQK + d] = orc_round_bf16(yd[d]);
            const uint16_t *vr = v + (r * hkv + h) * ORC_DV;
            for (int d = 0; d < ORC_DV; ++d)
                v_out[(r * hkv + h) * ORC_DV + d] = orc_round_bf16(orc_bf16(vr[d]) * value_scale);
        }
    }
}

/*
 * One sequence, one layer.
 *
 *   q      [nq][hq][192]  raw bf16 queries at positions qpos[nq]
 *   k      [nk][hkv][192] raw bf16 keys;   row r holds position k0 + r
 *   v      [nk][hkv][128] raw bf16 values; row r holds position k0 + r
 *   window 0 for a full-attention layer, else the window length (128)
 *   sinks  [hq] sink logits (windowed layers) or NULL (no sink term)
 *   out    [nq][hq][128]  fp64 attention output
 *   stats  [nq][hq][2]    (m, Z): the max used and the full denominator
 *                         sum_j e^{s_j-m} (+ e^{sink-m}); may be NULL
 *
 * Keys outside rows 0..nk-1 simply do not exist for this call: the caller
 * passes every key the definition wants (positions max(0,p-W+1)..p for a
 * windowed layer, 0..p for a full one) or, to test a property of the math,
 * a subset of them.  Returns 0, or -1 on a bad argument.
 */
int orc_attend_seq(const uint16_t *q, const int64_t *qpos, int64_t nq, int hq,
                   const uint16_t *k, const uint16_t *v, int64_t k0, int64_t nk, int hkv,
                   double theta, double value_scale, double softmax_scale, int64_t window,
                   const double *sinks, double *out, double *stats, int nthreads) {
    if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || nq < 0 || nk < 0) return -1;
    const int group = hq / hkv;

    /* k' = rope(k) and v' = v * value_scale for every key row, fp64. */
    double *kr = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1) * hkv * ORC_DQK);
    double *vr = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1) * hkv * ORC_DV);
    if (!kr || !vr) { free(kr); free(vr); return -1; }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t r = 0; r < nk; ++r) {
        double cs[2 * ORC_HALF], xd[ORC_DQK];
        orc_rope_cos_sin(theta, k0 + r, cs);
        for (int h = 0; h < hkv; ++h) {
            for (int d = 0; d < ORC_DQK; ++d) xd[d] = orc_bf16(k[(r * hkv + h) * ORC_DQK + d]);
            orc_rope_apply(xd, cs, kr + (r * hkv + h) * ORC_DQK);
            for (int d = 0; d < ORC_DV; ++d)
                vr[(r * hkv + h) * ORC_DV + d] = orc_bf16(v[(r * hkv + h) * ORC_DV + d]) * value_scale;
        }
    }

    const int64_t rows = nq * hq;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t row = 0; row < rows; ++row) {
        const int64_t i = row / hq;
        const int h = (int)(row % hq);
        const int kvh = h / group;
        const int64_t p = qpos[i];
        double cs[2 * ORC_HALF], xd[ORC_DQK], qr[ORC_DQK];
        orc_rope_cos_sin(theta, p, cs);
        for (int d = 0; d < ORC_DQK; ++d) xd[d] = orc_bf16(q[(i * hq + h) * ORC_DQK + d]);
        orc_rope_apply(xd, cs, qr);

        /* key positions in J(p), intersected with the rows given */
        int64_t lo = window > 0 ? p - window + 1 : 0;
        if (lo < k0) lo = k0;
        int64_t hi = p;
        if (hi > k0 + nk - 1) hi = k0 + nk - 1;

        /* pass 1: logits and their max (the sink takes part in the max) */
        double m = -INFINITY;
        if (sinks) m = sinks[h];
        for (int64_t j = lo; j <= hi; ++j) {
            const double *kk = kr + ((j - k0) * hkv + kvh) * ORC_DQK;
            double s = 0.0;
            for (int d = 0; d < ORC_DQK; ++d) s += qr[d] * kk[d];
            s *= softmax_scale;
            if (s > m) m = s;
        }
        /* pass 2: numerator and denominator */
        double z = 0.0, acc[ORC_DV];
        for (int d = 0; d < ORC_DV; ++d) acc[d] = 0.0;
        if (sinks) z += exp(sinks[h] - m);
        for (int64_t j = lo; j <= hi; ++j) {
            const double *kk = kr + ((j - k0) * hkv + kvh) * ORC_DQK;
            double s = 0.0;
            for (int d = 0; d < ORC_DQK; ++d) s += qr[d] * kk[d];
            s *= softmax_scale;
            double e = exp(s - m);
            z += e;
            const double *vv = vr + ((j - k0) * hkv + kvh) * ORC_DV;
            for (int d = 0; d < ORC_DV; ++d) acc[d] += e * vv[d];
        }
        double *o = out + (i * hq + h) * ORC_DV;
        for (int d = 0; d < ORC_DV; ++d) o[d] = z > 0.0 ? acc[d] / z : 0.0;
        if (stats) {
            stats[(i * hq + h) * 2] = m;
            stats[(i * hq + h) * 2 + 1] = z;
        }
    }
    free(kr);
    free(vr);
    return 0;
}

/* Threads OpenMP will use for a parallel region (1 without OpenMP). */
int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
