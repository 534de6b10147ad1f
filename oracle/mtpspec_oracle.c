/*
 * mtpspec oracle: a plain, slow, double-precision CPU statement of what the MTP
 * speculative-decoding hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  It is loaded by the test suite, by the package's smoke
 * check and by the benchmark's CPU-baseline leg and reference arm; the product library
 * never links, loads or calls it, and the two share no code (no headers, helpers or
 * tables).
 *
 * Sources, cited by page title and section:
 *  [HB] "14. MTP: speculative decoding with the built-in draft head" (Transformer by
 *       Hand, stage 2): "The draft head" (the MTP module: two RMSNorms, concatenation
 *       with the embedding first, fc = Linear(2H, H, bias=False)) and "The speculative
 *       decoding loop (greedy version)" (accept a draft when it equals the main
 *       model's argmax, else take the main model's own token).
 *  [DL] "The decoding loop and MTP" (agent-loop-visualizer docs): "Why a hand-written
 *       decoding loop" (temperature, then top-k, then top-p, then sample; argmax takes
 *       the lower id on ties) and "MTP speculative decoding" items 2-3 (first rejected
 *       guess replaced, later guesses dropped, one extra token when all guesses hold;
 *       a guess is kept with its probability and otherwise the token is drawn from the
 *       other candidates).
 *  [ZH] "MPT (MTP, Multi-Token Prediction) 原理详解": section 二.2 (enorm/hnorm, concat,
 *       eh_proj), section 三 stage 3 (greedy and rejection-sampling verification),
 *       stage 4 (1 to D+1 tokens per verification), section 四 (worked example).
 *  [PX] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 *       SC'11: the Philox4x32-10 counter-based generator.
 *
 * Readings where the pages are silent or garbled (each is restated in the design notes):
 *  - RMSNorm is x * 1/sqrt(mean(x^2) + eps) * w, and the normalised activations are
 *    rounded to bf16 before the projection, as a bf16 module would store them.
 *  - top-k keeps every value >= the k-th largest (ties at the boundary all kept);
 *    top-p keeps a token when the filtered mass of strictly larger logits is < p.
 *  - rejection-sampling residual is normalize(max(0, p_target - p_draft)); the page
 *    prints max(0, 1 - P_target/P_draft), which is not a distribution over tokens.
 *  - uniforms: Philox4x32-10, key = (seed lo, seed hi), counter = (row, position, 0, 0);
 *    U_acc from output word 0, U_smp from word 1, U = (2*(w >> 9) + 1) * 2^-24.
 *  - draws use the inverse CDF in ascending token-id order.
 *  - a temperature of 0 makes a row greedy: it takes the greedy rule and reports
 *    p_target = [d == argmax], p_draft = 1 (the greedy drafter's point mass).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_OK = 0, ORC_ERR_ARG = -1, ORC_ERR_DTYPE = -2, ORC_ERR_NAN = -7, ORC_ERR_NOMEM = -8 };
enum { ORC_STATUS_BAD_DRAFT_ID = 1 };

/* ------------------------------------------------------------------ value access */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double logit_at(const void *base, int dt, int64_t i)
{
    if (dt == ORC_F32)
        return (double)((const float *)base)[i];
    return bf16_bits_to_double(((const uint16_t *)base)[i]);
}

/* Round a double to the nearest bfloat16 (ties to even) and return its bit pattern.
 * bfloat16 keeps 8 significant bits and float's exponent range; its subnormal
 * quantum is 2^-133. */
uint16_t orc_double_to_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;      /* quantum of an 8-significant-bit number in that binade */
    if (q < -133)
        q = -133;
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* ------------------------------------------------------------------ Philox4x32-10 [PX] */

/* One Philox4x32 bijection with 10 rounds.  Each round multiplies words 0 and 2 by the
 * two round multipliers, swaps the halves and mixes in the key; the key is bumped by the
 * two Weyl constants between rounds (constants as published with the algorithm). */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    const uint64_t mul0 = 0xD2511F53u, mul1 = 0xCD9E8D57u;
    const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = mul0 * (uint64_t)c0;
        uint64_t p1 = mul1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += weyl0;
        k1 += weyl1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Map a 32-bit word to an odd multiple of 2^-24 in (0, 1); exactly representable in
 * float and double. */
static double word_to_uniform(uint32_t w)
{
    return (double)(2u * (w >> 9) + 1u) * ldexp(1.0, -24);
}

/* The two uniforms of verification unit (row, position): U_acc for the accept test,
 * U_smp for the draw at that position. */
void orc_uniforms(uint64_t seed, uint64_t row, uint32_t pos, double *u_acc, double *u_smp)
{
    uint32_t ctr[4] = {(uint32_t)row, pos, 0u, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t o[4];
    orc_philox4x32_10(ctr, key, o);
    *u_acc = word_to_uniform(o[0]);
    *u_smp = word_to_uniform(o[1]);
}

/* ------------------------------------------------------------------ argmax [DL] */

/* Index of the largest logit, the lowest index among equal maxima ("takes the lower
 * id", [DL] "Why a hand-written decoding loop").  -inf is an ordinary value, so an
 * all -inf row gives 0.  Returns -1 for V < 1 and -2 if a NaN is present. */
int64_t orc_argmax(const void *x, int dt, int64_t V)
{
    if (V < 1)
        return -1;
    int64_t best = 0;
    double bv = logit_at(x, dt, 0);
    if (isnan(bv))
        return -2;
    for (int64_t i = 1; i < V; ++i) {
        double v = logit_at(x, dt, i);
        if (isnan(v))
            return -2;
        if (v > bv) {
            bv = v;
            best = i;
        }
    }
    return best;
}

/* Greedy draft ([HB] "The draft head": draft = argmax of the draft logits; [ZH] 三
 * stages 1-2, greedy sample of each draft step): one argmax per row of [M, V]. */
int orc_greedy_draft(const void *logits, int dt, int64_t M, int64_t V, int32_t *ids)
{
    if (dt != ORC_F32 && dt != ORC_BF16)
        return ORC_ERR_DTYPE;
    if (M < 0 || V < 1 || (M > 0 && (!logits || !ids)))
        return ORC_ERR_ARG;
    size_t es = dt == ORC_F32 ? 4 : 2;
    for (int64_t r = 0; r < M; ++r) {
        int64_t a = orc_argmax((const char *)logits + (size_t)r * (size_t)V * es, dt, V);
        if (a < 0)
            return ORC_ERR_NAN;
        ids[r] = (int32_t)a;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ greedy verify */

/* Greedy verification ([HB] greedy loop; [ZH] 三 stage 3 "greedy strategy", stage 4;
 * [DL] item 2).  Row b has target logits T[b, 0..D, :] over the D+1 positions
 * [bonus, d_0 .. d_{D-1}] and drafts d[b, 0..D-1].  a = the first j with
 * d_j != argmax T[b, j] (D if none); the row emits d_0 .. d_{a-1} then argmax T[b, a]
 * (the correction, or the bonus when a = D); -1 pads to D+1.  An id outside [0, V)
 * never equals an argmax, so it is rejected, and it sets ORC_STATUS_BAD_DRAFT_ID. */
int orc_verify_greedy(const void *T, int dt, const int32_t *d, int64_t B, int32_t D, int64_t V,
                      int32_t *out, int32_t *num_accepted, int32_t *status)
{
    if (dt != ORC_F32 && dt != ORC_BF16)
        return ORC_ERR_DTYPE;
    if (B < 0 || D < 1 || V < 1)
        return ORC_ERR_ARG;
    size_t es = dt == ORC_F32 ? 4 : 2;
    int32_t st = 0;
    for (int64_t b = 0; b < B; ++b) {
        const char *rowT = (const char *)T + (size_t)b * (size_t)(D + 1) * (size_t)V * es;
        int32_t a = D;
        for (int32_t j = 0; j < D; ++j) {
            int32_t dj = d[b * D + j];
            if (dj < 0 || (int64_t)dj >= V)
                st |= ORC_STATUS_BAD_DRAFT_ID;
        }
        for (int32_t j = 0; j < D; ++j) {
            int64_t g = orc_argmax(rowT + (size_t)j * (size_t)V * es, dt, V);
            if (g < 0)
                return ORC_ERR_NAN;
            if ((int64_t)d[b * D + j] != g) {
                a = j;
                break;
            }
        }
        int64_t last = orc_argmax(rowT + (size_t)a * (size_t)V * es, dt, V);
        if (last < 0)
            return ORC_ERR_NAN;
        for (int32_t j = 0; j <= D; ++j)
            out[b * (D + 1) + j] = -1;
        for (int32_t j = 0; j < a; ++j)
            out[b * (D + 1) + j] = d[b * D + j];
        out[b * (D + 1) + a] = (int32_t)last;
        num_accepted[b] = a;
    }
    if (status)
        *status |= st;
    return ORC_OK;
}

/* ------------------------------------------------------------------ filtering [DL] */

typedef struct {
    double v;
    int64_t i;
} orc_vi;

static int orc_vi_desc(const void *pa, const void *pb)
{
    const orc_vi *a = (const orc_vi *)pa, *b = (const orc_vi *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

/* The sampling distribution of one logit row under temperature tau > 0, then top-k,
 * then top-p, "in turn" ([DL] "Why a hand-written decoding loop"):
 *   - top-k is on for 1 <= k < V: keep every logit >= the k-th largest one;
 *   - weights w_i = exp((x_i - max) / tau) over the kept set;
 *   - top-p is on for p < 1: keep a token when the normalised weight of the kept
 *     tokens with strictly larger logits is < p (the largest logits always stay);
 *   - the result is renormalised over what is left.
 * Writes the unnormalised kept weights to w[V], support membership to in[V] (a kept
 * token whose weight underflows is still in the support), their sum to *Z and the row
 * maximum to *mx.  A row whose logits are all -inf is a point mass on id 0, its
 * argmax.  *margin_p (if given) receives the distance from p of the two masses that
 * decide the top-p boundary (+inf when top-p is off).
 *
 * For the parity checker: the top-p rule walks groups of equal logits from the top, and
 * group g (1-based) stays when the mass S_g strictly above it is < p.  force_groups >= 1
 * keeps exactly the first force_groups groups of the top-k set instead (as a computation
 * whose masses are off by less than delta might); cuts (if given) receives the number of
 * groups the rule keeps and the smallest and largest counts that such a computation can
 * reach: g with S_g < p + delta and S_{g+1} >= p - delta (S of one past the last group
 * is 1).  With top-p off all three are the group count. */
static int orc_filter_weights_cut(const void *x, int dt, int64_t V, double tau, int32_t k,
                                  double p, int64_t force_groups, double delta, double *w,
                                  unsigned char *in, double *Z, double *mx, double *margin_p,
                                  int64_t *cuts)
{
    if (margin_p)
        *margin_p = INFINITY;
    if (cuts)
        cuts[0] = cuts[1] = cuts[2] = 1;
    orc_vi *s = (orc_vi *)malloc((size_t)V * sizeof(orc_vi));
    if (!s)
        return ORC_ERR_NOMEM;
    double m = -INFINITY;
    for (int64_t i = 0; i < V; ++i) {
        s[i].v = logit_at(x, dt, i);
        s[i].i = i;
        if (isnan(s[i].v)) {
            free(s);
            return ORC_ERR_NAN;
        }
        if (s[i].v > m)
            m = s[i].v;
    }
    *mx = m;
    for (int64_t i = 0; i < V; ++i) {
        w[i] = 0.0;
        in[i] = 0;
    }
    if (m == -INFINITY) {
        w[0] = 1.0;
        in[0] = 1;
        *Z = 1.0;
        free(s);
        return ORC_OK;
    }
    qsort(s, (size_t)V, sizeof(orc_vi), orc_vi_desc);

    /* top-k: the threshold is the k-th largest value, counting repeats */
    double theta = -INFINITY;
    if (k >= 1 && (int64_t)k < V)
        theta = s[k - 1].v;

    int64_t kept = 0; /* kept entries form a prefix of the sorted order */
    double z = 0.0;
    while (kept < V && s[kept].v >= theta) {
        double wi = exp((s[kept].v - m) / tau);
        w[s[kept].i] = wi;
        in[s[kept].i] = 1;
        z += wi;
        ++kept;
    }

    if (p < 1.0) {
        /* walk groups of equal logits from the top; S = normalised mass strictly above */
        double above = 0.0;
        int64_t g = 0, gi = 0, cut = -1, rule = 1, glo = -1, ghi = 1;
        while (g < kept) {
            int64_t h = g;
            double gm = 0.0;
            while (h < kept && s[h].v == s[g].v) {
                gm += w[s[h].i];
                ++h;
            }
            ++gi;
            double S = above / z;
            if (S < p + delta)
                ghi = gi;
            if (glo < 0 && ((above + gm) / z >= p - delta || h == kept))
                glo = gi;
            int keep = S < p;
            if (keep)
                rule = gi;
            if (force_groups >= 1)
                keep = gi <= force_groups;
            if (keep && cut < 0) {
                above += gm;
                if (margin_p && force_groups < 1) {
                    double mk = p - S; /* how far the kept group was from dropping */
                    double md = fabs(above / z - p); /* mass that the next group would see */
                    double mm = mk < md ? mk : md;
                    *margin_p = mm;
                }
            } else {
                if (cut < 0)
                    cut = g;
                above += gm;
            }
            g = h;
            if (cut >= 0 && S >= p && above / z >= p + delta && glo >= 0)
                break;
        }
        if (cuts) {
            cuts[0] = rule;
            cuts[1] = glo;
            cuts[2] = ghi;
        }
        if (cut >= 0) {
            for (int64_t t = cut; t < kept; ++t) {
                w[s[t].i] = 0.0;
                in[s[t].i] = 0;
            }
            kept = cut;
        }
        z = 0.0;
        for (int64_t t = 0; t < kept; ++t)
            z += w[s[t].i];
    } else if (cuts) {
        int64_t ng = 0;
        for (int64_t t = 0; t < kept; ++t)
            if (t == 0 || s[t].v != s[t - 1].v)
                ++ng;
        cuts[0] = cuts[1] = cuts[2] = ng;
    }
    *Z = z;
    free(s);
    return ORC_OK;
}

static int orc_filter_weights(const void *x, int dt, int64_t V, double tau, int32_t k, double p,
                              double *w, unsigned char *in, double *Z, double *mx, double *margin_p)
{
    return orc_filter_weights_cut(x, dt, V, tau, k, p, -1, 0.0, w, in, Z, mx, margin_p, NULL);
}

/* Normalised filtered probabilities of one row (see orc_filter_weights). */
int orc_filter(const void *x, int dt, int64_t V, double tau, int32_t k, double p, double *prob,
               double *margin_p)
{
    if (dt != ORC_F32 && dt != ORC_BF16)
        return ORC_ERR_DTYPE;
    if (V < 1 || !(tau > 0.0) || !(p > 0.0))
        return ORC_ERR_ARG;
    double Z, m;
    unsigned char *in = (unsigned char *)malloc((size_t)V);
    if (!in)
        return ORC_ERR_NOMEM;
    int rc = orc_filter_weights(x, dt, V, tau, k, p, prob, in, &Z, &m, margin_p);
    free(in);
    if (rc != ORC_OK)
        return rc;
    for (int64_t i = 0; i < V; ++i)
        prob[i] /= Z;
    return ORC_OK;
}

/* ------------------------------------------------------------------ draws */

/* Inverse-CDF draw over non-negative weights in ascending id order: the smallest i with
 * C(i) = sum_{y <= i} w_y > u * sum(w); if rounding leaves none, the largest i with
 * w_i > 0.  *margin receives min(u*S - C(i-1), C(i) - u*S) / S.  For the parity checker
 * nb (if given) receives those two distances apart, (u*S - C(i-1)) / S and
 * (C(i) - u*S) / S, and the nearest ids below and above i with positive weight (-1 if
 * none): the tokens a draw whose sums are off by less than the distance would give. */
static int64_t orc_inverse_cdf_nb(const double *w, int64_t V, double u, double *margin,
                                  double *nb)
{
    double S = 0.0;
    for (int64_t i = 0; i < V; ++i)
        S += w[i];
    double t = u * S;
    double c = 0.0;
    int64_t tok = -1;
    double lo = 0.0, hi = 0.0;
    for (int64_t i = 0; i < V; ++i) {
        double prev = c;
        c += w[i];
        if (c > t) {
            double a = (t - prev) / S, b = (c - t) / S;
            if (margin)
                *margin = a < b ? a : b;
            lo = a;
            hi = b;
            tok = i;
            break;
        }
    }
    if (tok < 0) {
        if (margin)
            *margin = 0.0;
        for (int64_t i = V - 1; i >= 0; --i)
            if (w[i] > 0.0) {
                tok = i;
                break;
            }
        if (tok < 0)
            tok = 0;
    }
    if (nb) {
        int64_t pv = -1, nx = -1;
        for (int64_t i = tok - 1; i >= 0; --i)
            if (w[i] > 0.0) {
                pv = i;
                break;
            }
        for (int64_t i = tok + 1; i < V; ++i)
            if (w[i] > 0.0) {
                nx = i;
                break;
            }
        nb[0] = lo;
        nb[1] = hi;
        nb[2] = (double)pv;
        nb[3] = (double)nx;
    }
    return tok;
}

/* ------------------------------------------------------------------ sampling verify */

/* Everything one verification unit (row b, position j) decides, given its uniforms. */
typedef struct {
    int32_t accept;      /* position j < D: the draft held */
    double pt, pd;       /* p_j(d_j), q_j(d_j) */
    double ratio;        /* p/q of the accept test (NAN when the test needs no ratio) */
    double acc_margin;   /* |U_acc - p/q| (+inf when no ratio is formed) */
    double mp_t, mp_q;   /* top-p margins of the target and draft rows */
    int64_t token;       /* the draw (at a rejection or at the bonus position), or -1 */
    double cdf_margin;   /* its inverse-CDF margin */
    double nb[4];        /* its distances to the neighbouring cells and their ids */
    int64_t cut_t[3], cut_q[3]; /* top-p group counts: the rule's, the smallest, the largest */
} orc_unit_result;

/* One unit of speculative-sampling verification ([ZH] 三 stage 3 "rejection sampling";
 * [DL] "MTP speculative decoding" items 2-3).  rowT / rowQ are T[b, j] and Q[b, j] (rowQ
 * NULL: a one-hot draft, q_j the point mass on d_j).  is_bonus: position D, whose token is
 * drawn from p_D.  Otherwise the accept test of d_j, and, if the draft is rejected and
 * want_draw is set, the draw from normalize(max(0, p_j - q_j)) (from p_j when that
 * residual is identically 0).  gt / gq force the top-p group counts of the two rows (-1:
 * the rule); delta is the window of the reported alternative counts.  w_draw (if given,
 * [V]) receives the unnormalised weights of the draw. */
static int orc_unit(const char *rowT, const char *rowQ, int dt, int64_t V, int32_t dj, double tb,
                    int32_t kb, double pb, double ua, double us, int is_bonus, int want_draw,
                    int64_t gt, int64_t gq, double delta, double *wp, double *wq, double *wr,
                    unsigned char *inp, unsigned char *inq, double *w_draw, orc_unit_result *o)
{
    double Zp, Zq, mp, mq, xp, xq;
    o->accept = 0;
    o->pt = o->pd = 0.0;
    o->ratio = NAN;
    o->acc_margin = INFINITY;
    o->mp_t = o->mp_q = INFINITY;
    o->token = -1;
    o->cdf_margin = INFINITY;
    for (int t = 0; t < 4; ++t)
        o->nb[t] = t < 2 ? INFINITY : -1.0;
    for (int t = 0; t < 3; ++t)
        o->cut_t[t] = o->cut_q[t] = 0;
    int rc = orc_filter_weights_cut(rowT, dt, V, tb, kb, pb, gt, delta, wp, inp, &Zp, &xp, &mp,
                                    o->cut_t);
    if (rc != ORC_OK)
        return rc;
    o->mp_t = mp;
    if (is_bonus) {
        double dm;
        o->token = orc_inverse_cdf_nb(wp, V, us, &dm, o->nb);
        o->cdf_margin = dm;
        if (w_draw)
            memcpy(w_draw, wp, (size_t)V * sizeof(double));
        return ORC_OK;
    }
    if (rowQ) {
        rc = orc_filter_weights_cut(rowQ, dt, V, tb, kb, pb, gq, delta, wq, inq, &Zq, &xq, &mq,
                                    o->cut_q);
        if (rc != ORC_OK)
            return rc;
        o->mp_q = mq;
    } else { /* one-hot draft: q_j = 1 at d_j, 0 elsewhere */
        for (int64_t i = 0; i < V; ++i) {
            wq[i] = 0.0;
            inq[i] = 0;
        }
        if (dj >= 0 && (int64_t)dj < V) {
            wq[dj] = 1.0;
            inq[dj] = 1;
        }
        Zq = 1.0;
        xq = 0.0;
    }
    int valid = dj >= 0 && (int64_t)dj < V;
    double pt = valid ? wp[dj] / Zp : 0.0;
    double pd = valid ? wq[dj] / Zq : 0.0;
    o->pt = pt;
    o->pd = pd;
    int accept;
    if (!valid || !inp[dj]) {
        accept = 0;
    } else if (!inq[dj]) {
        accept = 1;
    } else {
        /* p/q written with both row maxima factored out, so that it does not
         * underflow when both probabilities are tiny; a row of all -inf is a
         * point mass, whose probability is exact */
        double ratio;
        if (!rowQ || xp == -INFINITY || xq == -INFINITY) {
            ratio = pt / pd;
        } else {
            double xt = logit_at(rowT, dt, dj);
            double xd = logit_at(rowQ, dt, dj);
            ratio = exp(((xt - xp) - (xd - xq)) / tb) * (Zq / Zp);
        }
        accept = ua <= ratio;
        o->ratio = ratio;
        o->acc_margin = fabs(ua - ratio);
    }
    o->accept = accept;
    if (!accept && want_draw) {
        /* residual draw at the first rejection */
        double R = 0.0;
        for (int64_t i = 0; i < V; ++i) {
            double r = wp[i] / Zp - wq[i] / Zq;
            wr[i] = r > 0.0 ? r : 0.0;
            R += wr[i];
        }
        double dm;
        int64_t tok;
        if (R > 0.0)
            tok = orc_inverse_cdf_nb(wr, V, us, &dm, o->nb);
        else
            tok = orc_inverse_cdf_nb(wp, V, us, &dm, o->nb);
        o->token = tok;
        o->cdf_margin = dm;
        if (w_draw)
            memcpy(w_draw, R > 0.0 ? wr : wp, (size_t)V * sizeof(double));
    }
    return ORC_OK;
}

/* One unit with explicit uniforms, for the tests: the exact-enumeration pin integrates
 * over (u_acc, u_smp), and the parity checker evaluates the alternatives a computation off
 * by less than delta could take (gt / gq: forced top-p group counts, -1 for the rule).
 * Outputs: dres[8] = accept, p, q, ratio, |U_acc - ratio|, top-p margin of T, of Q, the
 * draw's inverse-CDF margin; dnb[4] = the draw's distances to its cell's edges and the
 * neighbouring ids; ires[7] = token (-1: no draw), the cut counts of T (rule, lowest,
 * highest) and of Q; w_draw [V] (optional) = the draw's unnormalised weights. */
int orc_verify_unit(const void *Trow, const void *Qrow, int dt, int64_t V, int32_t dj, double tau,
                    int32_t k, double p, double ua, double us, int32_t is_bonus, int32_t want_draw,
                    int64_t gt, int64_t gq, double delta, double *dres, double *dnb, int64_t *ires,
                    double *w_draw)
{
    if (dt != ORC_F32 && dt != ORC_BF16)
        return ORC_ERR_DTYPE;
    if (V < 1 || !Trow || !(tau > 0.0) || !(p > 0.0) || !dres || !dnb || !ires)
        return ORC_ERR_ARG;
    double *wp = (double *)malloc((size_t)V * sizeof(double) * 3);
    unsigned char *inp = (unsigned char *)malloc((size_t)V * 2);
    if (!wp || !inp) {
        free(wp);
        free(inp);
        return ORC_ERR_NOMEM;
    }
    orc_unit_result o;
    int rc = orc_unit((const char *)Trow, (const char *)Qrow, dt, V, dj, tau, k, p, ua, us,
                      is_bonus, want_draw, gt, gq, delta, wp, wp + V, wp + 2 * V, inp, inp + V,
                      w_draw, &o);
    free(wp);
    free(inp);
    if (rc != ORC_OK)
        return rc;
    dres[0] = o.accept;
    dres[1] = o.pt;
    dres[2] = o.pd;
    dres[3] = o.ratio;
    dres[4] = o.acc_margin;
    dres[5] = o.mp_t;
    dres[6] = o.mp_q;
    dres[7] = o.cdf_margin;
    for (int t = 0; t < 4; ++t)
        dnb[t] = o.nb[t];
    ires[0] = o.token;
    for (int t = 0; t < 3; ++t) {
        ires[1 + t] = o.cut_t[t];
        ires[4 + t] = o.cut_q[t];
    }
    return ORC_OK;
}

/* Speculative-sampling verification ([ZH] 三 stage 3 "rejection sampling", stage 4;
 * [DL] "MTP speculative decoding" items 2-3).  For row b with temperature tau_b > 0
 * and positions j = 0..D:
 *   p_j = filtered distribution of T[b, j];  q_j = filtered distribution of Q[b, j] (j < D)
 *   position j < D accepts d_j iff d_j is in the support of p_j and (d_j is outside the
 *       support of q_j, or U_acc(b, j) <= p_j(d_j) / q_j(d_j));  an id outside [0, V)
 *       is rejected;
 *   a = the first rejected position (D if none);
 *   a < D: the token at a is drawn from normalize(max(0, p_a - q_a)) with U_smp(b, a)
 *          (from p_a when that residual is identically 0);
 *   a = D: the bonus token is drawn from p_D with U_smp(b, D).
 * tau_b = 0 makes row b greedy (orc_verify_greedy's rule).  top_k / top_p may be NULL
 * (off).  Q may be NULL: a one-hot draft, q_j the point mass on d_j (a greedy drafter),
 * so that d_j is accepted iff U_acc <= p_j(d_j), q_j(d_j) = 1, and the residual is p_a
 * with d_a removed.  row0 offsets the Philox row counter (the rows passed are rows row0.. of a
 * larger batch).  out[B, D+1] (-1 padded), num_accepted[B]; p_target / p_draft [B, D]
 * receive p_j(d_j), q_j(d_j).  margins (optional) [B, D+1, 4] receive per unit:
 * |U_acc - p/q|, the top-p margin of T, of Q, and the draw's inverse-CDF margin
 * (+inf where not applicable). */
int orc_verify_sample(const void *T, const void *Q, int dt, const int32_t *d, const float *tau,
                      const int32_t *top_k, const float *top_p, uint64_t seed, int64_t row0,
                      int64_t B, int32_t D, int64_t V, int32_t *out, int32_t *num_accepted,
                      double *p_target, double *p_draft, int32_t *status, double *margins)
{
    if (dt != ORC_F32 && dt != ORC_BF16)
        return ORC_ERR_DTYPE;
    if (B < 0 || D < 1 || V < 1 || row0 < 0)
        return ORC_ERR_ARG;
    if (B == 0)
        return ORC_OK;
    if (!T || !d || !tau || !out || !num_accepted)
        return ORC_ERR_ARG;
    size_t es = dt == ORC_F32 ? 4 : 2;
    double *wp = (double *)malloc((size_t)V * sizeof(double) * 3);
    unsigned char *inp = (unsigned char *)malloc((size_t)V * 2);
    if (!wp || !inp) {
        free(wp);
        free(inp);
        return ORC_ERR_NOMEM;
    }
    double *wq = wp + V, *wr = wq + V;
    unsigned char *inq = inp + V;
    int32_t st = 0;
    int rc = ORC_OK;

    for (int64_t b = 0; b < B && rc == ORC_OK; ++b) {
        const char *rowT = (const char *)T + (size_t)b * (size_t)(D + 1) * (size_t)V * es;
        const char *rowQ = Q ? (const char *)Q + (size_t)b * (size_t)D * (size_t)V * es : NULL;
        double tb = (double)tau[b];
        int32_t kb = top_k ? top_k[b] : 0;
        double pb = top_p ? (double)top_p[b] : 1.0;
        if (!(tb >= 0.0) || !(pb > 0.0)) {
            rc = ORC_ERR_ARG;
            break;
        }
        double *mg = margins ? margins + (size_t)b * (size_t)(D + 1) * 4 : NULL;
        if (mg)
            for (int32_t t = 0; t < (D + 1) * 4; ++t)
                mg[t] = INFINITY;
        for (int32_t j = 0; j < D; ++j) {
            int32_t dj = d[b * D + j];
            if (dj < 0 || (int64_t)dj >= V)
                st |= ORC_STATUS_BAD_DRAFT_ID;
        }

        if (tb == 0.0) { /* greedy row */
            int32_t a = D;
            int64_t g_at_a = -1;
            for (int32_t j = 0; j <= D; ++j) {
                int64_t g = orc_argmax(rowT + (size_t)j * (size_t)V * es, dt, V);
                if (g < 0) {
                    rc = ORC_ERR_NAN;
                    break;
                }
                if (j < D) {
                    int32_t dj = d[b * D + j];
                    int valid = dj >= 0 && (int64_t)dj < V;
                    if (p_target)
                        p_target[b * D + j] = (valid && dj == g) ? 1.0 : 0.0;
                    if (p_draft)
                        p_draft[b * D + j] = valid ? 1.0 : 0.0;
                    if (a == D && (int64_t)dj != g)
                        a = j;
                }
                if (j == a && g_at_a < 0)
                    g_at_a = g;
            }
            if (rc != ORC_OK)
                break;
            for (int32_t j = 0; j <= D; ++j)
                out[b * (D + 1) + j] = -1;
            for (int32_t j = 0; j < a; ++j)
                out[b * (D + 1) + j] = d[b * D + j];
            out[b * (D + 1) + a] = (int32_t)g_at_a;
            num_accepted[b] = a;
            continue;
        }

        /* sampling row: accept tests at every position j < D; the draw at the first
         * rejection */
        int32_t a = D;
        for (int32_t j = 0; j < D && rc == ORC_OK; ++j) {
            double ua, us;
            orc_uniforms(seed, (uint64_t)(row0 + b), (uint32_t)j, &ua, &us);
            orc_unit_result o;
            rc = orc_unit(rowT + (size_t)j * (size_t)V * es,
                          rowQ ? rowQ + (size_t)j * (size_t)V * es : NULL, dt, V, d[b * D + j],
                          tb, kb, pb, ua, us, 0, a == D, -1, -1, 0.0, wp, wq, wr, inp, inq, NULL,
                          &o);
            if (rc != ORC_OK)
                break;
            if (p_target)
                p_target[b * D + j] = o.pt;
            if (p_draft)
                p_draft[b * D + j] = o.pd;
            if (mg) {
                mg[j * 4 + 0] = o.acc_margin;
                mg[j * 4 + 1] = o.mp_t;
                mg[j * 4 + 2] = o.mp_q;
            }
            if (!o.accept && a == D) {
                a = j;
                if (mg)
                    mg[j * 4 + 3] = o.cdf_margin;
                for (int32_t t = 0; t <= D; ++t)
                    out[b * (D + 1) + t] = -1;
                for (int32_t t = 0; t < a; ++t)
                    out[b * (D + 1) + t] = d[b * D + t];
                out[b * (D + 1) + a] = (int32_t)o.token;
                num_accepted[b] = a;
            }
        }
        if (rc != ORC_OK)
            break;
        if (a == D) { /* every draft held: bonus token from position D */
            double ua, us;
            orc_uniforms(seed, (uint64_t)(row0 + b), (uint32_t)D, &ua, &us);
            orc_unit_result o;
            rc = orc_unit(rowT + (size_t)D * (size_t)V * es, NULL, dt, V, -1, tb, kb, pb, ua, us,
                          1, 1, -1, -1, 0.0, wp, wq, wr, inp, inq, NULL, &o);
            if (rc != ORC_OK)
                break;
            if (mg) {
                mg[D * 4 + 1] = o.mp_t;
                mg[D * 4 + 3] = o.cdf_margin;
            }
            for (int32_t t = 0; t < D; ++t)
                out[b * (D + 1) + t] = d[b * D + t];
            out[b * (D + 1) + D] = (int32_t)o.token;
            num_accepted[b] = D;
        }
    }
    free(wp);
    free(inp);
    if (status)
        *status |= st;
    return rc;
}

/* ------------------------------------------------------------------ draft input [HB][ZH] */

/* RMSNorm of one H-vector with the pages' module layout ([HB] "The draft head":
 * RMSNorm(H, eps); [ZH] 二.2 step 2): out_i = bf16(v_i * r * w_i), r = 1/sqrt(mean(v^2)+eps). */
static void orc_rmsnorm_bf16(const uint16_t *v, const uint16_t *w, int64_t H, double eps,
                             double *out)
{
    double ss = 0.0;
    for (int64_t i = 0; i < H; ++i) {
        double x = bf16_bits_to_double(v[i]);
        ss += x * x;
    }
    double r = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t i = 0; i < H; ++i) {
        double y = bf16_bits_to_double(v[i]) * r * bf16_bits_to_double(w[i]);
        out[i] = bf16_bits_to_double(orc_double_to_bf16(y));
    }
}

/* The draft head's input stage ([HB] "The draft head": fc(cat(norm(e_{t+1}), norm(h_t)));
 * [ZH] 二.2 steps 2-3: eh_proj(cat(enorm(embeds), hnorm(hidden)))).  For each token t:
 * x = [enorm(e_t); hnorm(h_t)] (embedding first, 2H values), y_t = W x with W [H, 2H]
 * row-major (out x in, no bias), accumulated in double and returned before any output
 * rounding.  xn (optional) [M, 2H] receives the bf16 bits of x. */
int orc_draft_input(const uint16_t *e, const uint16_t *h, const uint16_t *we, const uint16_t *wh,
                    const uint16_t *W, int64_t M, int64_t H, double eps, double *y, uint16_t *xn)
{
    if (M < 0 || H < 1 || !(eps >= 0.0))
        return ORC_ERR_ARG;
    double *x = (double *)malloc((size_t)(2 * H) * sizeof(double));
    if (!x)
        return ORC_ERR_NOMEM;
    for (int64_t t = 0; t < M; ++t) {
        orc_rmsnorm_bf16(e + t * H, we, H, eps, x);
        orc_rmsnorm_bf16(h + t * H, wh, H, eps, x + H);
        if (xn)
            for (int64_t i = 0; i < 2 * H; ++i)
                xn[t * 2 * H + i] = orc_double_to_bf16(x[i]);
        for (int64_t o = 0; o < H; ++o) {
            const uint16_t *wrow = W + o * 2 * H;
            double acc = 0.0;
            for (int64_t i = 0; i < 2 * H; ++i)
                acc += bf16_bits_to_double(wrow[i]) * x[i];
            y[t * H + o] = acc;
        }
    }
    free(x);
    return ORC_OK;
}

/* Selected outputs y[tok[i], col[i]] of orc_draft_input, one at a time, for checks at
 * sizes where the full product is too slow on the host. */
int orc_draft_input_at(const uint16_t *e, const uint16_t *h, const uint16_t *we,
                       const uint16_t *wh, const uint16_t *W, int64_t M, int64_t H, double eps,
                       const int64_t *tok, const int64_t *col, int64_t n, double *y)
{
    if (M < 1 || H < 1 || n < 0 || !(eps >= 0.0))
        return ORC_ERR_ARG;
    double *x = (double *)malloc((size_t)(2 * H) * sizeof(double));
    if (!x)
        return ORC_ERR_NOMEM;
    int64_t cur = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (tok[i] < 0 || tok[i] >= M || col[i] < 0 || col[i] >= H) {
            free(x);
            return ORC_ERR_ARG;
        }
        if (tok[i] != cur) {
            cur = tok[i];
            orc_rmsnorm_bf16(e + cur * H, we, H, eps, x);
            orc_rmsnorm_bf16(h + cur * H, wh, H, eps, x + H);
        }
        const uint16_t *wrow = W + col[i] * 2 * H;
        double acc = 0.0;
        for (int64_t k = 0; k < 2 * H; ++k)
            acc += bf16_bits_to_double(wrow[k]) * x[k];
        y[i] = acc;
    }
    free(x);
    return ORC_OK;
}

/* ------------------------------------------------------------------ draft output layer [HB][ZH] */

/* Logits of the draft head's output layer for selected tokens ([HB] "The draft head": the
 * block's output goes through a normalisation and the output layer shared with the main
 * model; [ZH] 二.1 shared_head shares the main model's lm_head, 三 stage 1
 * compute_logits).  For token t = tok[i]: x = hidden[t] (bf16 [H]), replaced by its
 * RMSNorm with norm_w (bf16 result, the input stage's rule) when norm_w is given;
 * logits[i, v] = sum_k W[v, k] x_k in double for W [V, H] row-major (out x in, no bias).
 * absdot (optional) [n, V] receives sum_k |W[v, k] x_k|, the scale of the rounding error
 * a lower-precision sum of the same products can make. */
int orc_lm_head_logits(const uint16_t *hidden, const uint16_t *norm_w, double eps,
                       const uint16_t *W, int64_t M, int64_t H, int64_t V, const int64_t *tok,
                       int64_t n, double *logits, double *absdot)
{
    if (M < 0 || H < 1 || V < 1 || n < 0 || !(eps >= 0.0) || (n > 0 && (!hidden || !W || !tok || !logits)))
        return ORC_ERR_ARG;
    double *x = (double *)malloc((size_t)H * sizeof(double));
    if (!x)
        return ORC_ERR_NOMEM;
    for (int64_t i = 0; i < n; ++i) {
        if (tok[i] < 0 || tok[i] >= M) {
            free(x);
            return ORC_ERR_ARG;
        }
        const uint16_t *h = hidden + tok[i] * H;
        if (norm_w)
            orc_rmsnorm_bf16(h, norm_w, H, eps, x);
        else
            for (int64_t k = 0; k < H; ++k)
                x[k] = bf16_bits_to_double(h[k]);
        for (int64_t v = 0; v < V; ++v) {
            const uint16_t *wrow = W + v * H;
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < H; ++k) {
                double pr = bf16_bits_to_double(wrow[k]) * x[k];
                acc += pr;
                aacc += fabs(pr);
            }
            logits[i * V + v] = acc;
            if (absdot)
                absdot[i * V + v] = aacc;
        }
    }
    free(x);
    return ORC_OK;
}

/* The greedy draft from the output layer ([HB] "The draft head" and the greedy loop: the
 * draft is the argmax of the draft logits; [DL] "Why a hand-written decoding loop": argmax
 * takes the lower id on ties; [ZH] 三 stage 1 greedy sample): ids[t] = the lowest v with
 * the largest logit of token t, for every token; maxv (optional) = that logit. */
int orc_lm_head_greedy(const uint16_t *hidden, const uint16_t *norm_w, double eps,
                       const uint16_t *W, int64_t M, int64_t H, int64_t V, int32_t *ids,
                       double *maxv)
{
    if (M < 0 || H < 1 || V < 1 || V > 2147483647 || (M > 0 && !ids))
        return ORC_ERR_ARG;
    double *lg = (double *)malloc((size_t)V * sizeof(double));
    if (!lg)
        return ORC_ERR_NOMEM;
    for (int64_t t = 0; t < M; ++t) {
        int rc = orc_lm_head_logits(hidden, norm_w, eps, W, M, H, V, &t, 1, lg, NULL);
        if (rc != ORC_OK) {
            free(lg);
            return rc;
        }
        int64_t best = 0;
        for (int64_t v = 1; v < V; ++v)
            if (lg[v] > lg[best])
                best = v;
        ids[t] = (int32_t)best;
        if (maxv)
            maxv[t] = lg[best];
    }
    free(lg);
    return ORC_OK;
}

/* ------------------------------------------------------------------ post-verify state [HB] */

/* Snapshot before verification ([HB] "Rolling back" and the snapshot step of the decoding
 * loop: a KV cache only needs its length, which the caller keeps; the linear attention's
 * memory tables and convolution windows are copied): backup[b] = state[b] for each of B
 * rows of row_bytes bytes. */
int orc_state_snapshot(const uint8_t *state, uint8_t *backup, int64_t B, int64_t row_bytes)
{
    if (B < 0 || row_bytes < 0 || (B > 0 && row_bytes > 0 && (!state || !backup)))
        return ORC_ERR_ARG;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t i = 0; i < row_bytes; ++i)
            backup[b * row_bytes + i] = state[b * row_bytes + i];
    return ORC_OK;
}

/* Fix-up after verification ([HB] "Rolling back" and the loop's hit / miss branches; [ZH]
 * 三 stage 4; the accepted count a comes from the verifier).  The verify forward appended
 * D + 1 positions (the carried-in token and the D drafts) after kv_before[b] positions.
 *  - a == D (hit): every appended position stays: kv_len = kv_before + D + 1, the state is
 *    kept, nothing is recomputed.
 *  - a < D (miss), with a recurrent state (row_bytes > 0): the memory tables have absorbed
 *    rejected drafts and cannot be undone, so the row goes back to its snapshot: state =
 *    backup, kv_len = kv_before (a truncation), and the carried-in token and the a
 *    accepted drafts (recompute = 1 + a) must pass the model again.
 *  - a < D without a recurrent state (row_bytes == 0): attention keys of kept positions do
 *    not depend on later ones, so kv_len = kv_before + 1 + a and nothing is recomputed.
 *  - on a miss, the draft head's own KV length is cut to the main model's:
 *    draft_kv_len = min(draft_kv_len, kv_len).
 * A row with a outside [0, D] is left untouched and sets ORC_STATUS_BAD_PARAM (2). */
int orc_state_fixup(const int32_t *num_accepted, int32_t D, const int32_t *kv_before,
                    int32_t *kv_len, uint8_t *state, const uint8_t *backup, int64_t B,
                    int64_t row_bytes, int32_t *draft_kv_len, int32_t *recompute,
                    int32_t *status)
{
    if (B < 0 || D < 1 || row_bytes < 0)
        return ORC_ERR_ARG;
    if (B > 0 && (!num_accepted || !kv_before || !kv_len || (row_bytes > 0 && (!state || !backup))))
        return ORC_ERR_ARG;
    int32_t st = 0;
    for (int64_t b = 0; b < B; ++b) {
        const int32_t a = num_accepted[b];
        if (a < 0 || a > D) {
            st |= 2;
            continue;
        }
        const int miss = a < D;
        int32_t kv, rc = 0;
        if (!miss) {
            kv = kv_before[b] + D + 1;
        } else if (row_bytes > 0) {
            for (int64_t i = 0; i < row_bytes; ++i)
                state[b * row_bytes + i] = backup[b * row_bytes + i];
            kv = kv_before[b];
            rc = 1 + a;
        } else {
            kv = kv_before[b] + 1 + a;
        }
        kv_len[b] = kv;
        if (recompute)
            recompute[b] = rc;
        if (draft_kv_len && miss && draft_kv_len[b] > kv)
            draft_kv_len[b] = kv;
    }
    if (status)
        *status |= st;
    return ORC_OK;
}

/* ------------------------------------------------------------------ draft steps [ZH][HB] */

/* D serial draft steps of the draft head ([ZH] 三 stage 1 and stage 2: the bonus token and
 * the main model's hidden state start the chain; each step embeds the previous token,
 * runs the head and greedy-samples the next draft, and feeds that token and the head's
 * hidden state to the next step; 二.2 step 1: the input embedding at position 0 is zeroed;
 * [HB] "The draft head").  The head's decoder block is not modelled: its output is its
 * input (a stub), so a step is
 *     e   = embed[ids] (a zero row where positions[t] + step == 0)
 *     y   = bf16(eh_proj(cat(enorm(e), hnorm(h))))     (orc_draft_input, then rounded)
 *     ids = argmax over v of lm_head(norm(y))          (orc_lm_head_greedy's rule)
 *     h   = y
 * embed [V, H] and lm_head_w [V, H] bf16; positions may be NULL (no mask); norm_w may be
 * NULL (no final norm).  draft_ids [M, D]; hidden_out (optional) [D, M, H] bf16 bits of
 * each step's y.  An id outside [0, V) embeds as a zero row and sets status bit 1. */
int orc_draft_steps(const uint16_t *embed, const int32_t *next_ids, const int32_t *positions,
                    const uint16_t *hidden, const uint16_t *enorm_w, const uint16_t *hnorm_w,
                    const uint16_t *eh_proj_w, const uint16_t *norm_w, const uint16_t *lm_head_w,
                    double eps, int64_t M, int64_t H, int64_t V, int32_t D, int32_t *draft_ids,
                    uint16_t *hidden_out, int32_t *status)
{
    if (M < 0 || H < 1 || V < 1 || D < 1 || !(eps >= 0.0))
        return ORC_ERR_ARG;
    if (M == 0)
        return ORC_OK;
    if (!embed || !next_ids || !hidden || !enorm_w || !hnorm_w || !eh_proj_w || !lm_head_w || !draft_ids)
        return ORC_ERR_ARG;
    uint16_t *e = (uint16_t *)calloc((size_t)(M * H), sizeof(uint16_t));
    uint16_t *h = (uint16_t *)malloc((size_t)(M * H) * sizeof(uint16_t));
    int32_t *ids = (int32_t *)malloc((size_t)M * sizeof(int32_t));
    double *y = (double *)malloc((size_t)(M * H) * sizeof(double));
    if (!e || !h || !ids || !y) {
        free(e); free(h); free(ids); free(y);
        return ORC_ERR_NOMEM;
    }
    memcpy(h, hidden, (size_t)(M * H) * sizeof(uint16_t));
    memcpy(ids, next_ids, (size_t)M * sizeof(int32_t));
    int32_t st = 0;
    int rc = ORC_OK;
    for (int32_t k = 0; k < D && rc == ORC_OK; ++k) {
        for (int64_t t = 0; t < M; ++t) {
            const int masked = positions && (int64_t)positions[t] + k == 0;
            const int bad = ids[t] < 0 || ids[t] >= V;
            if (bad)
                st |= 1;
            for (int64_t i = 0; i < H; ++i)
                e[t * H + i] = (masked || bad) ? 0 : embed[(int64_t)ids[t] * H + i];
        }
        rc = orc_draft_input(e, h, enorm_w, hnorm_w, eh_proj_w, M, H, eps, y, NULL);
        if (rc != ORC_OK)
            break;
        for (int64_t i = 0; i < M * H; ++i)
            h[i] = orc_double_to_bf16(y[i]);
        if (hidden_out)
            memcpy(hidden_out + (int64_t)k * M * H, h, (size_t)(M * H) * sizeof(uint16_t));
        rc = orc_lm_head_greedy(h, norm_w, eps, lm_head_w, M, H, V, ids, NULL);
        for (int64_t t = 0; t < M && rc == ORC_OK; ++t)
            draft_ids[t * D + k] = ids[t];
    }
    free(e); free(h); free(ids); free(y);
    if (status)
        *status |= st;
    return rc;
}

/* The k largest logits of the draft output layer, for a drafter that proposes several
 * candidates ([HB] "The draft head" and [ZH] 三 stage 1: the output layer's logits; [DL]
 * "Why a hand-written decoding loop": top-k keeps the k largest, and a tie goes to the
 * lower id).  For each token t, ids[t, 0..k-1] lists the ids of the k largest logits in
 * decreasing order, equal logits in increasing id order; vals (optional) their logits. */
int orc_lm_head_topk(const uint16_t *hidden, const uint16_t *norm_w, double eps,
                     const uint16_t *W, int64_t M, int64_t H, int64_t V, int32_t k, int32_t *ids,
                     double *vals)
{
    if (M < 0 || H < 1 || V < 1 || V > 2147483647 || k < 1 || k > V || (M > 0 && !ids))
        return ORC_ERR_ARG;
    double *lg = (double *)malloc((size_t)V * sizeof(double));
    unsigned char *taken = (unsigned char *)malloc((size_t)V);
    if (!lg || !taken) {
        free(lg);
        free(taken);
        return ORC_ERR_NOMEM;
    }
    for (int64_t t = 0; t < M; ++t) {
        int rc = orc_lm_head_logits(hidden, norm_w, eps, W, M, H, V, &t, 1, lg, NULL);
        if (rc != ORC_OK) {
            free(lg);
            free(taken);
            return rc;
        }
        memset(taken, 0, (size_t)V);
        for (int32_t r = 0; r < k; ++r) {  /* k selections of the largest remaining logit */
            int64_t best = -1;
            for (int64_t v = 0; v < V; ++v)
                if (!taken[v] && (best < 0 || lg[v] > lg[best]))
                    best = v;
            taken[best] = 1;
            ids[t * k + r] = (int32_t)best;
            if (vals)
                vals[t * k + r] = lg[best];
        }
    }
    free(lg);
    free(taken);
    return ORC_OK;
}
