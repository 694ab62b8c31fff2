/*
 * moe_oracle.c -- CPU oracle for the fused MoE hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only through the seeded input generators.
 *
 * It is written to be checked by eye against the definition of a top-k
 * mixture-of-experts layer, not to be fast:
 *   - one token at a time, one routed slot at a time, plain loops;
 *   - every floating-point sum of the experts' arithmetic in double (fp64);
 *   - the decisions that pick an integer (which experts a token goes to, which
 *     e4m3 code a value gets) are taken in fp32, the precision the CUDA
 *     kernels take them in, so that ids and codes can be compared bit for bit.
 *
 * Passages followed (web pages on the subject, cited by title and section):
 *   [MK]  "vllm/model_executor/layers/fused_moe/modular_kernel.py"
 *         (vllm-cpu 0.11.0.post2 diff view):
 *         - module comment: [Router] -> [Quantize-Dispatch] ->
 *           [Permute-Experts-Unpermute] -> [Combine];
 *         - _moe_problem_size: E, M, N, K, topk; w1 is (E, 2N, K) with the
 *           gated pair stacked along its rows, w2 is (E, K, N); Standard
 *           format a1 (M, K), BatchedExperts format a1 (E, max_tokens, K);
 *         - ExpertTokensMetadata: per-expert token counts;
 *         - FusedMoEPrepareAndFinalize.prepare: quantisation happens before
 *           the experts run;
 *         - FusedMoEPermuteExpertsUnpermute.activation: a gated activation
 *           whose output is half as wide as its input (silu_and_mul);
 *         - FusedMoEPrepareAndFinalize.finalize: fused_expert_output has
 *           shape (M, topk, K); weights are applied and the topk slots are
 *           reduced into output (M, K).
 *   [WT]  "EP: CUDA-graph-safe HT internode dispatch+combine (worst-tokens
 *         mode)" (uccl pull request 7): a device int32[num_local_experts]
 *         count per expert, read by a masked grouped GEMM that only touches
 *         the first count rows of each expert's padded block.
 *
 * The pages do not spell out the router, the FP8 formula or which half of w1
 * is the gate; the readings taken here (named R1..R6, Q1..Q5, G1, G2, F1, B1,
 * B2 in the design notes) are:
 *   R1 softmax router: top-k on the raw logits (softmax is monotone), weight
 *      p_j = softmax(l)_j, renormalised over the chosen k when asked.
 *   R2 sigmoid grouped router: s_e = sigmoid(l_e + b_e); E experts in
 *      n_groups contiguous groups; group key = sum of the group's two largest
 *      s; keep the topk_groups best groups, then the topk best experts by s
 *      among them; weight s_j, renormalised when asked.  Experts are ranked
 *      by v_e = l_e + b_e (fp32), the order of the real-valued scores.
 *   R4 equal keys: the lower index wins (expert id, group id).
 *   R5 in a group key each s is the fp32 rounding of the fp64 value
 *      1/(1+exp(-(double)v)); the key is the fp32 add of the two.
 *   R6 ids in a row are in descending score order.
 *   P1 within one expert, pairs keep ascending pair order p = t*topk + j.
 *   Q1 FP8 group quant: s = max(amax, 1e-12) / 448 in fp32,
 *      q = e4m3(x / s) with round-to-nearest-even, saturating at +-448.
 *   G1 rows [0, N) of w1[e] are the gate (SiLU applied), rows [N, 2N) the up
 *      projection; G2 silu(z) = z / (1 + exp(-z)).
 *   Q5 optional requantisation of the hidden row h in 128-wide groups.
 *   F1 the topk slots are summed in slot order j = 0..topk-1.
 *   B1 batched rows r >= count[e] are neither read nor written.
 *   B3 expert_map (FusedMoEModularKernel.forward): global -> local expert
 *      ids of this shard, -1 = not here (the pair adds nothing);
 *      apply_router_weight_on_input (prepare, forward; topk 1): the router
 *      weight multiplies the expert's input, not its output.
 *   Q6 per_act_token_quant with per_out_ch_quant (the quant config's
 *      properties on FusedMoEPermuteExpertsUnpermute): the Q1 rule with one
 *      group per row -- one scale per token over its K values, one scale per
 *      output channel (row) of w1 and w2.  The hidden row h is kept in
 *      bf16 between the GEMMs (the activations' dtype) and quantised per
 *      token over its N values before the second GEMM, as prepare
 *      quantises the input of the experts.
 *   Q7 per-tensor activation scales (per_act_token_quant off, no block
 *      shape): the Q1 rule with one group holding the whole tensor -- one
 *      scale for the layer's input x (all M tokens) and one for H (every
 *      routed pair's hidden row, kept in bf16 as in Q6); weights as in Q6
 *      (per-tensor weight scales are equal per-row scales).
 *   Q8 static per-tensor activation scales (the quant config's a1_scale and
 *      a2_scale, FusedMoEPrepareAndFinalize.prepare): as Q7, but the scale of
 *      x and the scale of H are given instead of taken from the tensors'
 *      maxima; q = e4m3(v / scale), saturating at +-448 like every code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ORC_FP8: 1 x 128 activation groups, 128 x 128 weight blocks (Q1, Q2);
 * ORC_FP8_CHANNEL: one scale per token and one per weight row (Q6);
 * ORC_FP8_TENSOR: one scale per activation tensor, one per weight row (Q7) */
enum { ORC_BF16 = 0, ORC_FP8 = 1, ORC_FP8_CHANNEL = 2, ORC_FP8_TENSOR = 3 };
enum { ORC_SOFTMAX = 0, ORC_SIGMOID = 1 };
/* FusedMoEPermuteExpertsUnpermute.activation: "silu" -> silu_and_mul,
 * "gelu" -> gelu_and_mul */
enum { ORC_SILU = 0, ORC_GELU = 1 };

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the top half of an IEEE binary32: widening is exact. */
static double bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* e4m3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, subnormals when the exponent field is 0, no infinities, and the
 * single NaN pattern S.1111.111.  Largest finite magnitude 1.75 * 2^8 = 448. */
double orc_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int ex = (code >> 3) & 15;
    int man = code & 7;
    double v;
    if (ex == 15 && man == 7)
        return NAN;
    if (ex == 0)
        v = ldexp((double)man / 8.0, -6);
    else
        v = ldexp(1.0 + (double)man / 8.0, ex - 7);
    return sign ? -v : v;
}

/* orc_e4m3_value of every code, filled once before any parallel loop */
static double e4m3_table[256];
static void fill_e4m3_table(void)
{
    int c;
    for (c = 0; c < 256; ++c)
        e4m3_table[c] = orc_e4m3_value((uint8_t)c);
}

/* Round-to-nearest-even onto the e4m3 grid, saturating to +-448.  The
 * non-negative finite codes 0x00..0x7e are in increasing order of value, so
 * the nearest code is found by bisection for the last code whose value does
 * not exceed |x|, then a comparison with the next one; a tie (|x| exactly half
 * way) goes to the even code, the one whose mantissa ends in 0.  The sign is
 * carried separately, so negative values that round to zero give 0x80. */
uint8_t orc_e4m3_encode(float x)
{
    uint8_t sign;
    double a, dlo, dhi;
    int lo, hi, c;
    if (isnan(x))
        return 0x7f;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    lo = 0;    /* value(lo) <= a */
    hi = 0x7e; /* value(hi) >  a */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_e4m3_value((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    dlo = a - orc_e4m3_value((uint8_t)lo);
    dhi = orc_e4m3_value((uint8_t)hi) - a;
    if (dlo < dhi)
        c = lo;
    else if (dhi < dlo)
        c = hi;
    else
        c = (lo & 1) == 0 ? lo : hi;
    return (uint8_t)(sign | c);
}

/* Q1: scale of one group from its largest magnitude (fp32 arithmetic). */
static float group_scale(float amax)
{
    float m = amax > 1e-12f ? amax : 1e-12f;
    return m / 448.0f;
}

/* ------------------------------------------------------------------------ */
/* [Router] -- R1, R2, R4, R5, R6                                            */
/* ------------------------------------------------------------------------ */

/* R1 for one token.  ids[j], w[j] for j < topk. */
static void route_softmax_row(const float *l, int E, int topk, int renorm,
                              int32_t *ids, double *w)
{
    int j, e;
    float lmax = l[0];
    double denom = 0.0, sel = 0.0;
    char *taken = (char *)calloc((size_t)E, 1);
    for (e = 1; e < E; ++e)
        if (l[e] > lmax)
            lmax = l[e];
    for (e = 0; e < E; ++e)
        denom += exp((double)l[e] - (double)lmax);
    for (j = 0; j < topk; ++j) {
        int best = -1;
        for (e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || l[e] > l[best]) /* strict: lower id wins ties */
                best = e;
        }
        taken[best] = 1;
        ids[j] = best;
        w[j] = exp((double)l[best] - (double)lmax) / denom;
        sel += w[j];
    }
    if (renorm)
        for (j = 0; j < topk; ++j)
            w[j] /= sel;
    free(taken);
}

/* R5: the score a group key is built from -- the fp32 rounding of the fp64
 * value 1 / (1 + exp(-v)). */
static float sigmoid_score(float v)
{
    return (float)(1.0 / (1.0 + exp(-(double)v)));
}

/* R2 for one token.  The sigmoid is strictly increasing, so ranking experts
 * by their score is ranking them by v_e = l_e + b_e (an exact fp32 add);
 * experts are chosen on v, which keeps the order of the real-valued scores
 * (no ties made by rounding s to fp32).  A group's key is the fp32 sum of the
 * fp32 scores of its two largest v.
 * margin (optional) receives the fp64 gap between the last kept and the best
 * dropped group key (+inf without group limit): a tiny gap marks a token
 * whose group choice a last-bit difference in exp could flip. */
static void route_sigmoid_row(const float *l, const float *bias, int E,
                              int topk, int n_groups, int topk_groups,
                              int renorm, int32_t *ids, double *w,
                              double *margin)
{
    int gsz, g, e, j, i;
    float *v = (float *)malloc(sizeof(float) * (size_t)E);
    float *key;
    double *key64;
    char *gsel, *taken;
    double sel = 0.0, mg = INFINITY;

    if (n_groups < 1)
        n_groups = 1;
    if (topk_groups < 1 || topk_groups > n_groups)
        topk_groups = n_groups;
    gsz = E / n_groups;
    key = (float *)malloc(sizeof(float) * (size_t)n_groups);
    key64 = (double *)malloc(sizeof(double) * (size_t)n_groups);
    gsel = (char *)calloc((size_t)n_groups, 1);
    taken = (char *)calloc((size_t)E, 1);

    for (e = 0; e < E; ++e)
        v[e] = l[e] + (bias ? bias[e] : 0.0f);

    /* group key from the group's two largest v (one when the group has a
     * single expert); which of two equal v is "first" does not matter */
    for (g = 0; g < n_groups; ++g) {
        int a = -1, c = -1;
        for (i = 0; i < gsz; ++i) {
            e = g * gsz + i;
            if (a < 0 || v[e] > v[a]) {
                c = a;
                a = e;
            } else if (c < 0 || v[e] > v[c]) {
                c = e;
            }
        }
        if (c >= 0) {
            key[g] = sigmoid_score(v[a]) + sigmoid_score(v[c]);
            key64[g] = 1.0 / (1.0 + exp(-(double)v[a])) +
                       1.0 / (1.0 + exp(-(double)v[c]));
        } else {
            key[g] = sigmoid_score(v[a]);
            key64[g] = 1.0 / (1.0 + exp(-(double)v[a]));
        }
    }

    if (topk_groups < n_groups) {
        int last = -1;
        for (i = 0; i < topk_groups; ++i) {
            int best = -1;
            for (g = 0; g < n_groups; ++g) {
                if (gsel[g])
                    continue;
                if (best < 0 || key[g] > key[best])
                    best = g;
            }
            gsel[best] = 1;
            last = best;
        }
        for (g = 0; g < n_groups; ++g)
            if (!gsel[g] && key64[last] - key64[g] < mg)
                mg = key64[last] - key64[g];
    } else {
        for (g = 0; g < n_groups; ++g)
            gsel[g] = 1;
    }

    for (j = 0; j < topk; ++j) {
        int best = -1;
        for (e = 0; e < E; ++e) {
            if (taken[e] || !gsel[e / gsz])
                continue;
            if (best < 0 || v[e] > v[best])
                best = e;
        }
        taken[best] = 1;
        ids[j] = best;
        w[j] = 1.0 / (1.0 + exp(-(double)v[best]));
        sel += w[j];
    }
    if (renorm)
        for (j = 0; j < topk; ++j)
            w[j] /= sel;
    if (margin)
        *margin = mg;

    free(v);
    free(key);
    free(key64);
    free(gsel);
    free(taken);
}

/* [Router] over M tokens: logits (M, E) fp32, optional bias (E) fp32;
 * ids (M, topk) int32, w (M, topk) fp64, margin (M) fp64 or NULL. */
void orc_route(const float *logits, const float *bias, int M, int E, int topk,
               int score_fn, int n_groups, int topk_groups, int renorm,
               int32_t *ids, double *w, double *margin)
{
    int t;
    for (t = 0; t < M; ++t) {
        const float *l = logits + (size_t)t * E;
        if (score_fn == ORC_SOFTMAX) {
            route_softmax_row(l, E, topk, renorm, ids + (size_t)t * topk,
                              w + (size_t)t * topk);
            if (margin)
                margin[t] = INFINITY;
        } else {
            route_sigmoid_row(l, bias, E, topk, n_groups, topk_groups, renorm,
                              ids + (size_t)t * topk, w + (size_t)t * topk,
                              margin ? margin + t : NULL);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Counts and permutation -- ExpertTokensMetadata, "Permute" of             */
/* [Permute-Experts-Unpermute]; P1                                           */
/* ------------------------------------------------------------------------ */

/* The local expert of a routed (global) id -- the expert_map argument of
 * FusedMoEModularKernel.forward / FusedMoEPermuteExpertsUnpermute.apply maps
 * global expert ids to this expert-parallel shard's local ids.  map NULL:
 * the identity (E_global == E_local).  Returns the local id, -1 for an
 * expert that is not on this shard (map value -1: the pair is not computed
 * here), -2 for an id that is invalid (outside [0, E_global), or mapped
 * outside [0, E_local)). */
static int local_expert(int g, int E_global, const int32_t *map, int E_local)
{
    int l;
    if (g < 0 || g >= E_global)
        return -2;
    l = map ? map[g] : g;
    if (l == -1)
        return -1;
    if (l < 0 || l >= E_local)
        return -2;
    return l;
}

/* counts[l] = number of pairs p < P whose id maps to local expert l.
 * Returns how many ids were invalid (those pairs are left out, as are the
 * pairs of experts that are not local). */
int orc_count_mapped(const int32_t *ids, int P, int E_global,
                     const int32_t *map, int E_local, int32_t *counts)
{
    int p, bad = 0;
    memset(counts, 0, sizeof(int32_t) * (size_t)E_local);
    for (p = 0; p < P; ++p) {
        int l = local_expert(ids[p], E_global, map, E_local);
        if (l == -2)
            ++bad;
        if (l < 0)
            continue;
        counts[l] += 1;
    }
    return bad;
}

int orc_count(const int32_t *ids, int P, int E, int32_t *counts)
{
    return orc_count_mapped(ids, P, E, NULL, E, counts);
}

/* Stable counting sort of pair ids by (local) expert: offsets (E_local+1)
 * exclusive prefix sums of the counts; sorted[offsets[l] + r] = the r-th
 * pair (in ascending pair order) routed to l; inv[p] = its position, -1 for
 * a pair that is not computed here (invalid id, or an expert that is not
 * local). */
void orc_align_mapped(const int32_t *ids, int P, int E_global,
                      const int32_t *map, int E_local, int32_t *offsets,
                      int32_t *sorted, int32_t *inv)
{
    int p, e;
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E_local > 0 ? E_local : 1));
    orc_count_mapped(ids, P, E_global, map, E_local, cursor);
    offsets[0] = 0;
    for (e = 0; e < E_local; ++e)
        offsets[e + 1] = offsets[e] + cursor[e];
    for (e = 0; e < E_local; ++e)
        cursor[e] = offsets[e];
    for (p = 0; p < P; ++p) {
        int l = local_expert(ids[p], E_global, map, E_local);
        if (l < 0) {
            inv[p] = -1;
            continue;
        }
        sorted[cursor[l]] = p;
        inv[p] = cursor[l];
        cursor[l] += 1;
    }
    free(cursor);
}

void orc_align(const int32_t *ids, int P, int E, int32_t *offsets,
               int32_t *sorted, int32_t *inv)
{
    orc_align_mapped(ids, P, E, NULL, E, offsets, sorted, inv);
}

/* Gather: xperm[i] = x[sorted[i] / topk] for i < n_rows (rows of K doubles). */
void orc_permute_rows(const double *x, const int32_t *sorted, int n_rows,
                      int topk, int K, double *xperm)
{
    int i, k;
    for (i = 0; i < n_rows; ++i)
        for (k = 0; k < K; ++k)
            xperm[(size_t)i * K + k] = x[(size_t)(sorted[i] / topk) * K + k];
}

/* Unpermute + TopKWeightAndReduce: out[t] = sum_{j=0..topk-1}
 * w[t,j] * yperm[inv[t*topk+j]] in slot order (F1).  Pairs with inv < 0
 * contribute nothing. */
void orc_unpermute_reduce(const double *yperm, const int32_t *inv,
                          const double *w, int M, int topk, int K, double *out)
{
    int t, j, k;
    for (t = 0; t < M; ++t) {
        for (k = 0; k < K; ++k)
            out[(size_t)t * K + k] = 0.0;
        for (j = 0; j < topk; ++j) {
            int p = t * topk + j;
            if (inv[p] < 0)
                continue;
            for (k = 0; k < K; ++k)
                out[(size_t)t * K + k] +=
                    w[p] * yperm[(size_t)inv[p] * K + k];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* [Quantize-Prepare] -- Q1 and its 2-D block form for weights               */
/* ------------------------------------------------------------------------ */

/* x (M, K) bf16 -> q (M, K) e4m3 codes, scales (M, K / group) fp32.
 * row_w (M) or NULL: with apply_router_weight_on_input (prepare applies the
 * router weight to the activations before quantising), row t is first
 * multiplied by row_w[t] -- an fp32 product, the precision the codes are
 * decided in. */
void orc_quant_fp8_group_w(const uint16_t *x, const float *row_w, int M,
                           int K, int group, uint8_t *q, float *scales)
{
    int t, G = K / group;
    /* rows are independent: each one is quantised by one thread */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (t = 0; t < M; ++t) {
        int g, k;
        const float rw = row_w ? row_w[t] : 1.0f;
        for (g = 0; g < G; ++g) {
            const uint16_t *xg = x + (size_t)t * K + (size_t)g * group;
            float amax = 0.0f, s;
            for (k = 0; k < group; ++k) {
                float v = (float)fabs((float)bf16_value(xg[k]) * rw);
                if (v > amax)
                    amax = v;
            }
            s = group_scale(amax);
            scales[(size_t)t * G + g] = s;
            for (k = 0; k < group; ++k)
                q[(size_t)t * K + (size_t)g * group + k] =
                    orc_e4m3_encode(((float)bf16_value(xg[k]) * rw) / s);
        }
    }
}

void orc_quant_fp8_group(const uint16_t *x, int M, int K, int group,
                         uint8_t *q, float *scales)
{
    orc_quant_fp8_group_w(x, NULL, M, K, group, q, scales);
}

/* Q8: the codes of x (times row_w[t] in fp32 when given) with a given
 * scale: q = e4m3(v / scale), saturating. */
void orc_quant_fp8_tensor_static(const uint16_t *x, const float *row_w, int M,
                                 int K, float scale, uint8_t *q)
{
    int t, k;
    for (t = 0; t < M; ++t) {
        const float rw = row_w ? row_w[t] : 1.0f;
        for (k = 0; k < K; ++k)
            q[(size_t)t * K + k] =
                orc_e4m3_encode(((float)bf16_value(x[(size_t)t * K + k]) * rw) / scale);
    }
}

/* Q7: one group holding all M rows of x (times row_w[t] in fp32 when given):
 * *scale = max(amax, 1e-12) / 448, q = e4m3(v / scale). */
void orc_quant_fp8_tensor(const uint16_t *x, const float *row_w, int M, int K,
                          uint8_t *q, float *scale)
{
    int t, k;
    float amax = 0.0f, s;
    for (t = 0; t < M; ++t) {
        const float rw = row_w ? row_w[t] : 1.0f;
        for (k = 0; k < K; ++k) {
            float v = (float)fabs((float)bf16_value(x[(size_t)t * K + k]) * rw);
            if (v > amax)
                amax = v;
        }
    }
    s = group_scale(amax);
    *scale = s;
    for (t = 0; t < M; ++t) {
        const float rw = row_w ? row_w[t] : 1.0f;
        for (k = 0; k < K; ++k)
            q[(size_t)t * K + k] =
                orc_e4m3_encode(((float)bf16_value(x[(size_t)t * K + k]) * rw) / s);
    }
}

/* w (R, C) bf16 -> q (R, C) e4m3, scales (R / block, C / block) fp32; one
 * scale per block x block tile from the tile's largest magnitude. */
void orc_quant_fp8_block(const uint16_t *w, int R, int C, int block,
                         uint8_t *q, float *scales)
{
    int br, BR = R / block, BC = C / block;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (br = 0; br < BR; ++br) {
        int bc, r, c;
        for (bc = 0; bc < BC; ++bc) {
            float amax = 0.0f, s;
            for (r = br * block; r < (br + 1) * block; ++r)
                for (c = bc * block; c < (bc + 1) * block; ++c) {
                    float v = (float)fabs(bf16_value(w[(size_t)r * C + c]));
                    if (v > amax)
                        amax = v;
                }
            s = group_scale(amax);
            scales[(size_t)br * BC + bc] = s;
            for (r = br * block; r < (br + 1) * block; ++r)
                for (c = bc * block; c < (bc + 1) * block; ++c)
                    q[(size_t)r * C + c] = orc_e4m3_encode(
                        (float)bf16_value(w[(size_t)r * C + c]) / s);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* One expert on one row -- [Permute-Experts-Unpermute] apply: matmul,       */
/* act_mul, optional quant, matmul; G1, G2, Q5                               */
/* ------------------------------------------------------------------------ */

/* The weights of one run, one pointer per expert (NULL for an expert the
 * caller did not supply; using one is an error the caller must avoid).
 * dtype ORC_BF16: w1[e] (2N, K) and w2[e] (K, N) hold bf16 bits.  ORC_FP8:
 * they hold e4m3 codes, and w1s[e] (2N/128, K/128), w2s[e] (K/128, N/128)
 * hold the 128 x 128 block scales.  ORC_FP8_CHANNEL: e4m3 codes with one
 * scale per row, w1s[e] (2N), w2s[e] (K). */
typedef struct {
    int dtype, E, N, K;
    int act; /* ORC_SILU or ORC_GELU: the gated activation of the experts */
    const void *const *w1, *const *w2;
    const float *const *w1s, *const *w2s;
} orc_weights;

/* element (e, row, col) of a weight tensor (E, R, C), dequantised */
static double weight_at(const orc_weights *W, int which, int e, int row,
                        int col)
{
    int C = which == 1 ? W->K : W->N;
    size_t idx = (size_t)row * C + col;
    if (W->dtype == ORC_BF16) {
        const uint16_t *b = (const uint16_t *)(which == 1 ? W->w1[e] : W->w2[e]);
        return bf16_value(b[idx]);
    } else {
        const uint8_t *q = (const uint8_t *)(which == 1 ? W->w1[e] : W->w2[e]);
        const float *sc = which == 1 ? W->w1s[e] : W->w2s[e];
        size_t sidx = W->dtype == ORC_FP8_CHANNEL || W->dtype == ORC_FP8_TENSOR
                          ? (size_t)row
                          : (size_t)(row / 128) * (C / 128) + col / 128;
        return e4m3_table[q[idx]] * (double)sc[sidx];
    }
}

/* bf16 rounding (nearest, ties to even) of the fp32 rounding of v */
static double bf16_round(double v)
{
    float f = (float)v;
    uint32_t u;
    uint16_t h;
    memcpy(&u, &f, 4);
    h = (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
    return bf16_value(h);
}

/* h (N) = silu(x W1[e][0:N]^T) * (x W1[e][N:2N]^T); optional requant of h
 * (Q5: 128-wide groups of the fp32 h; Q6 for ORC_FP8_CHANNEL: h rounded to
 * bf16, then one group of N); y (K) = h W2[e]^T.  x is the (dequantised)
 * input row of K values. */
/* h (N) = act(x W1[e][0:N]^T) * (x W1[e][N:2N]^T) */
static void expert_h(const orc_weights *W, int e, const double *x, double *h)
{
    int n, k, N = W->N, K = W->K;
    for (n = 0; n < N; ++n) {
        double g = 0.0, u = 0.0;
        for (k = 0; k < K; ++k) {
            g += x[k] * weight_at(W, 1, e, n, k);
            u += x[k] * weight_at(W, 1, e, N + n, k);
        }
        if (W->act == ORC_GELU)
            h[n] = 0.5 * g * (1.0 + erf(g / sqrt(2.0))) * u; /* exact GELU */
        else
            h[n] = g / (1.0 + exp(-g)) * u;                  /* SiLU */
    }
}

/* y (K) = h W2[e]^T */
static void expert_y(const orc_weights *W, int e, const double *h, double *y)
{
    int n, k, N = W->N, K = W->K;
    for (k = 0; k < K; ++k) {
        double acc = 0.0;
        for (n = 0; n < N; ++n)
            acc += h[n] * weight_at(W, 2, e, k, n);
        y[k] = acc;
    }
}

static void expert_row(const orc_weights *W, int e, const double *x,
                       int requant_h, double *h, double *y)
{
    int n, N = W->N;
    expert_h(W, e, x, h);
    if (requant_h) {
        int gi, gw = W->dtype == ORC_FP8_CHANNEL ? N : 128;
        if (W->dtype == ORC_FP8_CHANNEL)
            for (n = 0; n < N; ++n)
                h[n] = bf16_round(h[n]);
        for (gi = 0; gi < N / gw; ++gi) {
            float amax = 0.0f, s;
            for (n = gi * gw; n < (gi + 1) * gw; ++n) {
                float v = (float)fabs((float)h[n]);
                if (v > amax)
                    amax = v;
            }
            s = group_scale(amax);
            for (n = gi * gw; n < (gi + 1) * gw; ++n)
                h[n] = orc_e4m3_value(orc_e4m3_encode((float)h[n] / s)) *
                       (double)s;
        }
    }
    expert_y(W, e, h, y);
}

/* Input row t of x (M, K) bf16 times `scale`, as the experts see it: the
 * product as is for bf16, or through Q1 (groups of 128, with the product
 * formed in fp32) for FP8, or through Q6 (one group of K) for
 * ORC_FP8_CHANNEL.  scale is 1 except with apply_router_weight_on_input. */
static void input_row_scaled(int dtype, const uint16_t *x, int t, int K,
                             double scale, double *xr)
{
    int k;
    const uint16_t *row = x + (size_t)t * K;
    if (dtype == ORC_BF16) {
        for (k = 0; k < K; ++k)
            xr[k] = bf16_value(row[k]) * scale;
    } else {
        float fs = (float)scale;
        int group = dtype == ORC_FP8_CHANNEL ? K : 128;
        uint8_t *q = (uint8_t *)malloc((size_t)K);
        float *s = (float *)malloc(sizeof(float) * (size_t)(K / group));
        orc_quant_fp8_group_w(row, &fs, 1, K, group, q, s);
        for (k = 0; k < K; ++k)
            xr[k] = orc_e4m3_value(q[k]) * (double)s[k / group];
        free(q);
        free(s);
    }
}

static void input_row(int dtype, const uint16_t *x, int t, int K, double *xr)
{
    input_row_scaled(dtype, x, t, K, 1.0, xr);
}

/* h and y of one expert on one row of x (bf16 bits); for checking the two
 * grouped GEMMs separately.  h (N), y (K) fp64. */
void orc_expert_row(int dtype, const uint16_t *x, int t, int e, int E, int N,
                    int K, const void *const *w1, const float *const *w1s,
                    const void *const *w2, const float *const *w2s,
                    int requant_h, double *h, double *y, int act)
{
    orc_weights W;
    double *xr = (double *)malloc(sizeof(double) * (size_t)K);
    fill_e4m3_table();
    W.dtype = dtype; W.E = E; W.N = N; W.K = K; W.act = act;
    W.w1 = w1; W.w2 = w2; W.w1s = w1s; W.w2s = w2s;
    input_row(dtype, x, t, K, xr);
    expert_row(&W, e, xr, requant_h, h, y);
    free(xr);
}

/* ------------------------------------------------------------------------ */
/* The layer, Standard format (M, K): for each listed token t,               */
/*   out[t] = sum_{j=0..topk-1} w[t,j] * expert_{ids[t,j]}(x[t])             */
/* -- FusedMoEModularKernel.forward with finalize's weight-and-reduce; F1    */
/* ------------------------------------------------------------------------ */

/* tokens (n_tok) lists which tokens to compute (NULL: all M, n_tok = M);
 * out (n_tok, K), ids_out (n_tok, topk), w_out (n_tok, topk) fp64.
 * Tokens are independent, so a listed subset is computed exactly as it
 * would be in a full run.  nthreads <= 0: the OpenMP default.
 * E is the number of routed (global) experts, the width of the logits.
 * expert_map (E) or NULL, E_local: the weights hold E_local experts; a pair
 * whose expert maps to -1 is not computed on this shard and adds nothing
 * (FusedMoEModularKernel.forward's expert_map).  weight_on_input
 * (apply_router_weight_on_input, meant for topk == 1): the router weight
 * multiplies the expert's input instead of its output,
 *   out[t] = sum_j expert(w[t,j] * x[t]). */
/* The layer with dynamic per-tensor activation scales (Q7).  The scale of H
 * spans every routed pair, so this takes two passes: first x's scale and
 * every local pair's hidden row (all M tokens, whatever `tokens` lists),
 * then the scale of H and the outputs of the listed tokens.  Arguments as
 * orc_moe_forward_ep. */
static void forward_tensor(const uint16_t *x, const float *logits,
                           const float *bias, int M, int K, int N, int E,
                           int topk, int score_fn, int n_groups,
                           int topk_groups, int renorm, int requant_h,
                           const int32_t *expert_map, int E_local,
                           int weight_on_input, const orc_weights *W,
                           const int32_t *tokens, int n_tok, int32_t *ids_out,
                           double *w_out, double *out)
{
    const size_t P = (size_t)M * topk;
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (P ? P : 1));
    double *w = (double *)malloc(sizeof(double) * (P ? P : 1));
    float *rw = (float *)malloc(sizeof(float) * (size_t)(M ? M : 1));
    uint8_t *xq = (uint8_t *)malloc((size_t)M * K + 1);
    double *h = (double *)malloc(sizeof(double) * (P * N + 1));
    char *local = (char *)malloc(P + 1);
    double *xr = (double *)malloc(sizeof(double) * (size_t)K);
    double *hq = (double *)malloc(sizeof(double) * (size_t)N);
    double *y = (double *)malloc(sizeof(double) * (size_t)K);
    float sx, sh = 1.0f, amax = 0.0f;
    int t, j, k, n, i;
    for (t = 0; t < M; ++t) {
        orc_route(logits + (size_t)t * E, bias, 1, E, topk, score_fn, n_groups,
                  topk_groups, renorm, ids + (size_t)t * topk,
                  w + (size_t)t * topk, NULL);
        rw[t] = (float)w[(size_t)t * topk]; /* weight on input: topk is 1 */
    }
    orc_quant_fp8_tensor(x, weight_on_input ? rw : NULL, M, K, xq, &sx);
    for (t = 0; t < M; ++t) {
        for (k = 0; k < K; ++k)
            xr[k] = orc_e4m3_value(xq[(size_t)t * K + k]) * (double)sx;
        for (j = 0; j < topk; ++j) {
            size_t p = (size_t)t * topk + j;
            int l = local_expert(ids[p], E, expert_map, E_local);
            local[p] = l >= 0;
            if (l < 0)
                continue;
            expert_h(W, l, xr, h + p * N);
            for (n = 0; n < N; ++n) {
                float v;
                h[p * N + n] = bf16_round(h[p * N + n]);
                v = (float)fabs((float)h[p * N + n]);
                if (v > amax)
                    amax = v;
            }
        }
    }
    if (requant_h)
        sh = group_scale(amax);
    if (!tokens)
        n_tok = M;
    for (i = 0; i < n_tok; ++i) {
        double *o = out + (size_t)i * K;
        t = tokens ? tokens[i] : i;
        for (k = 0; k < K; ++k)
            o[k] = 0.0;
        for (j = 0; j < topk; ++j) {
            size_t p = (size_t)t * topk + j;
            ids_out[(size_t)i * topk + j] = ids[p];
            w_out[(size_t)i * topk + j] = w[p];
            if (!local[p])
                continue;
            for (n = 0; n < N; ++n)
                hq[n] = requant_h ? orc_e4m3_value(orc_e4m3_encode(
                                        (float)h[p * N + n] / sh)) * (double)sh
                                  : h[p * N + n];
            expert_y(W, local_expert(ids[p], E, expert_map, E_local), hq, y);
            for (k = 0; k < K; ++k)
                o[k] += (weight_on_input ? 1.0 : w[p]) * y[k];
        }
    }
    free(ids); free(w); free(rw); free(xq); free(h); free(local);
    free(xr); free(hq); free(y);
}

/* The layer with static per-tensor activation scales (Q8): sx codes x, sh
 * codes H (each routed hidden row rounded to bf16 first, as in Q7).  No scale
 * depends on other tokens, so each listed token is computed on its own, in
 * the steps of the Q7 layer: its row of x (times its router weight in fp32
 * with weight_on_input) coded with sx, each local pair's hidden row rounded
 * to bf16 and (requant_h) coded with sh, the down projection, the weighted
 * sum in slot order.  Arguments as orc_moe_forward_ep. */
static void forward_tensor_static(const uint16_t *x, const float *logits,
                                  const float *bias, int K, int N, int E,
                                  int topk, int score_fn, int n_groups,
                                  int topk_groups, int renorm, int requant_h,
                                  const int32_t *expert_map, int E_local,
                                  int weight_on_input, const orc_weights *W,
                                  const int32_t *tokens, int n_tok,
                                  int32_t *ids_out, double *w_out, double *out,
                                  float sx, float sh, int nthreads)
{
    int i;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (i = 0; i < n_tok; ++i) {
        int t = tokens ? tokens[i] : i;
        int j, k, n;
        int32_t *ids = ids_out + (size_t)i * topk;
        double *w = w_out + (size_t)i * topk;
        uint8_t *xq = (uint8_t *)malloc((size_t)K);
        double *xr = (double *)malloc(sizeof(double) * (size_t)K);
        double *h = (double *)malloc(sizeof(double) * (size_t)N);
        double *y = (double *)malloc(sizeof(double) * (size_t)K);
        double *o = out + (size_t)i * K;
        float rw;
        orc_route(logits + (size_t)t * E, bias, 1, E, topk, score_fn, n_groups,
                  topk_groups, renorm, ids, w, NULL);
        rw = (float)w[0]; /* weight on input: topk is 1 */
        orc_quant_fp8_tensor_static(x + (size_t)t * K, weight_on_input ? &rw : NULL,
                                    1, K, sx, xq);
        for (k = 0; k < K; ++k) {
            xr[k] = orc_e4m3_value(xq[k]) * (double)sx;
            o[k] = 0.0;
        }
        for (j = 0; j < topk; ++j) {
            int l = local_expert(ids[j], E, expert_map, E_local);
            if (l < 0)
                continue;
            expert_h(W, l, xr, h);
            for (n = 0; n < N; ++n) {
                h[n] = bf16_round(h[n]);
                if (requant_h)
                    h[n] = orc_e4m3_value(orc_e4m3_encode((float)h[n] / sh)) * (double)sh;
            }
            expert_y(W, l, h, y);
            for (k = 0; k < K; ++k)
                o[k] += (weight_on_input ? 1.0 : w[j]) * y[k];
        }
        free(xq); free(xr); free(h); free(y);
    }
}

void orc_moe_forward_ep(const uint16_t *x, const float *logits,
                        const float *bias, int M, int K, int N, int E,
                        int topk, int score_fn, int n_groups, int topk_groups,
                        int renorm, int dtype, int requant_h,
                        const int32_t *expert_map, int E_local,
                        int weight_on_input, const void *const *w1,
                        const float *const *w1s, const void *const *w2,
                        const float *const *w2s, const int32_t *tokens,
                        int n_tok, int32_t *ids_out, double *w_out,
                        double *out, int nthreads, int act,
                        const float *static_scales)
{
    int i;
    orc_weights W;
    fill_e4m3_table();
    W.dtype = dtype; W.E = E_local; W.N = N; W.K = K; W.act = act;
    W.w1 = w1; W.w2 = w2; W.w1s = w1s; W.w2s = w2s;
    if (dtype == ORC_FP8_TENSOR && static_scales) {
        forward_tensor_static(x, logits, bias, K, N, E, topk, score_fn, n_groups,
                              topk_groups, renorm, requant_h, expert_map, E_local,
                              weight_on_input, &W, tokens, tokens ? n_tok : M,
                              ids_out, w_out, out, static_scales[0],
                              static_scales[1], nthreads);
        return;
    }
    if (dtype == ORC_FP8_TENSOR) {
        forward_tensor(x, logits, bias, M, K, N, E, topk, score_fn, n_groups,
                       topk_groups, renorm, requant_h, expert_map, E_local,
                       weight_on_input, &W, tokens, n_tok, ids_out, w_out, out);
        return;
    }
    if (!tokens)
        n_tok = M;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (i = 0; i < n_tok; ++i) {
        int t = tokens ? tokens[i] : i;
        int j, k;
        int32_t *ids = ids_out + (size_t)i * topk;
        double *w = w_out + (size_t)i * topk;
        double *xr = (double *)malloc(sizeof(double) * (size_t)K);
        double *h = (double *)malloc(sizeof(double) * (size_t)N);
        double *y = (double *)malloc(sizeof(double) * (size_t)K);
        double *o = out + (size_t)i * K;
        orc_route(logits + (size_t)t * E, bias, 1, E, topk, score_fn, n_groups,
                  topk_groups, renorm, ids, w, NULL);
        if (!weight_on_input)
            input_row(dtype, x, t, K, xr);
        for (k = 0; k < K; ++k)
            o[k] = 0.0;
        for (j = 0; j < topk; ++j) {
            int l = local_expert(ids[j], E, expert_map, E_local);
            if (l < 0)
                continue;
            if (weight_on_input) {
                /* the weight as the kernels hold it: fp32 */
                input_row_scaled(dtype, x, t, K, (double)(float)w[j], xr);
                expert_row(&W, l, xr, requant_h, h, y);
                for (k = 0; k < K; ++k)
                    o[k] += y[k];
            } else {
                expert_row(&W, l, xr, requant_h, h, y);
                for (k = 0; k < K; ++k)
                    o[k] += w[j] * y[k];
            }
        }
        free(xr);
        free(h);
        free(y);
    }
}

void orc_moe_forward(const uint16_t *x, const float *logits, const float *bias,
                     int M, int K, int N, int E, int topk, int score_fn,
                     int n_groups, int topk_groups, int renorm, int dtype,
                     int requant_h, const void *const *w1,
                     const float *const *w1s, const void *const *w2,
                     const float *const *w2s, const int32_t *tokens,
                     int n_tok, int32_t *ids_out, double *w_out, double *out,
                     int nthreads)
{
    orc_moe_forward_ep(x, logits, bias, M, K, N, E, topk, score_fn, n_groups,
                       topk_groups, renorm, dtype, requant_h, NULL, E, 0, w1,
                       w1s, w2, w2s, tokens, n_tok, ids_out, w_out, out,
                       nthreads, ORC_SILU, NULL);
}

/* ------------------------------------------------------------------------ */
/* BatchedExperts format (E, T, K) masked by per-expert counts -- [WT];      */
/* B1: y_b[e, r] = expert_e(x_b[e, r]) for r < min(count[e], T) only.        */
/* ------------------------------------------------------------------------ */

/* rows (n_rows, 2) lists (e, r) pairs to compute (NULL: every valid row of
 * every expert, in (e, r) order, n_rows ignored).  yb (E*T, K) fp64 is
 * written only at the computed rows.  Returns the number of rows computed. */
int orc_batched_experts(const uint16_t *xb, const int32_t *counts, int E,
                        int T, int N, int K, int dtype, int requant_h,
                        const void *const *w1, const float *const *w1s,
                        const void *const *w2, const float *const *w2s,
                        const int32_t *rows, int n_rows,
                        double *yb, int nthreads, int act)
{
    int e, i, n = 0;
    int32_t *list;
    orc_weights W;
    fill_e4m3_table();
    W.dtype = dtype; W.E = E; W.N = N; W.K = K; W.act = act;
    W.w1 = w1; W.w2 = w2; W.w1s = w1s; W.w2s = w2s;
    if (rows) {
        list = (int32_t *)rows;
        n = n_rows;
    } else {
        int total = 0, r;
        for (e = 0; e < E; ++e) {
            int c = counts[e] < 0 ? 0 : (counts[e] > T ? T : counts[e]);
            total += c;
        }
        list = (int32_t *)malloc(sizeof(int32_t) * 2 * (size_t)(total > 0 ? total : 1));
        for (e = 0; e < E; ++e) {
            int c = counts[e] < 0 ? 0 : (counts[e] > T ? T : counts[e]);
            for (r = 0; r < c; ++r) {
                list[2 * n] = e;
                list[2 * n + 1] = r;
                ++n;
            }
        }
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (i = 0; i < n; ++i) {
        int ee = list[2 * i], r = list[2 * i + 1];
        int c = counts[ee] < 0 ? 0 : (counts[ee] > T ? T : counts[ee]);
        double *xr, *h;
        if (r >= c)
            continue; /* B1: a padded row is never touched */
        xr = (double *)malloc(sizeof(double) * (size_t)K);
        h = (double *)malloc(sizeof(double) * (size_t)N);
        input_row(dtype, xb, ee * T + r, K, xr);
        expert_row(&W, ee, xr, requant_h, h, yb + ((size_t)ee * T + r) * K);
        free(xr);
        free(h);
    }
    if (!rows)
        free(list);
    return n;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
