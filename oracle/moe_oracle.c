/*
 * moe_oracle.c -- plain, slow, obviously correct fp64 CPU oracle for the
 * single-GPU Mixture-of-Experts FFN hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * bench's cpu_baseline / reference leg may load this library.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * What it computes, and the passages it follows:
 *   - top-k routing with fp32 logits and a softmax over the k selected logits
 *     ("[JAX] Expert Parallelism: JAX primitives + VJPs", squashed commit log:
 *     router logits promoted to fp32, fused_topk_with_score_function);
 *   - the expert-major permutation with -1 marking a dropped route
 *     ("Add MoE + expert-parallel Python API surface, PyTorch reference, and
 *     tests", Summary: routing, "-1 = dropped route"; _count_local_routes:
 *     other ids outside [0,E) are an error);
 *   - per-route SwiGLU experts silu(gate) * up, the down projection and the
 *     per-top-k weighted combine (same page, Summary: "local SwiGLU experts",
 *     "Form-A per-top-k combine");
 *   - the backward: re-dispatch dY along the forward routes, recompute SwiGLU
 *     from the bf16 fc1_c stash, wgrad/dgrad, scatter route gradients (same
 *     page, Summary: backward paragraph); zero wgrad for 0-token experts
 *     ("[JAX] Expert Parallelism", commit log: per-group zero-fill of wgrad);
 *   - MXFP8: E4M3 elements with one UE8M0 scale per 1x32 block along K
 *     (same cudnn-frontend page, BlockScaledTensor: block_size 32 for mxfp8).
 *
 * Arithmetic is double.  round_mode = 1 rounds to bf16 exactly where the
 * GPU path stores a bf16 tensor (h, the expert output y, out, dy_perm, dg/du,
 * dx; dx_perm and the weight gradients are fp32 on the path and are not
 * rounded here).  The rounding points of the forward are the benchmark
 * configuration's: h = bf16(silu(g) u) and y = bf16(h W_down), the pages'
 * expert outputs travelling in 2-byte slots ("[JAX] Expert Parallelism: JAX
 * primitives + VJPs", commit log: the fp32 island around silu and multiply
 * dropped, bf16 combine slots);
 * round_mode = 0 keeps every intermediate in double (used to pin the
 * formulas against fp64 autograd); round_mode = 2 rounds the stored
 * intermediates (h, y, dy_perm, dg/du) but returns the final
 * outputs (out, dx, dW) unrounded, so that a bf16 output of the GPU can be
 * compared with the exact value of the same arithmetic.  Readings of points the pages leave open
 * (tie-break, NaN order, MX scale rule) are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 bit pattern -> value (exact). */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> bf16 bit pattern, round to nearest even, overflow to inf.
 * bf16 has 8 significant bits and the fp32 exponent range. */
uint16_t oracle_double_to_bf16(double x)
{
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
    int lead = e - 1;
    int q = (lead < -126 ? -126 : lead) - 7;   /* quantum exponent */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r >= 0x1p128) return sign | 0x7F80;
    float f = (float)r;           /* exact: <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

static double bf(double x) { return oracle_bf16_to_double(oracle_double_to_bf16(x)); }
/* Rounding of a stored intermediate (round_mode 1 and 2) and of a final
 * output (round_mode 1 only: mode 2 returns the exact value of the final
 * sum, computed from intermediates rounded where the path stores them). */
static double rnd(double x, int round_mode) { return round_mode ? bf(x) : x; }
static double rnd_out(double x, int round_mode) { return round_mode == 1 ? bf(x) : x; }

/* OCP FP8 E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities, NaN = S.1111.111, largest finite 448 = S.1111.110. */
double oracle_e4m3_to_double(uint8_t c)
{
    int s = c >> 7, ex = (c >> 3) & 0xF, m = c & 7;
    if (ex == 0xF && m == 7) return NAN;
    double v = (ex == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), ex - 10);
    return s ? -v : v;
}

/* Round to nearest even onto the E4M3 grid, saturating finite values to
 * +-448 (the "satfinite" conversion). */
uint8_t oracle_double_to_e4m3(double x)
{
    if (isnan(x)) return 0x7F;
    uint8_t s = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0) return s | 0x7E;
    if (a == 0.0) return s;
    int e;
    frexp(a, &e);
    int lead = e - 1;
    int q = (lead < -6 ? -6 : lead) - 3;        /* 3 mantissa bits */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r > 448.0) return s | 0x7E;
    if (r < 0x1p-6) {                           /* subnormal (or 2^-6 itself) */
        int m = (int)ldexp(r, 9);               /* r = m * 2^-9, m in [0, 8] */
        return s | (uint8_t)m;
    }
    int ee;
    frexp(r, &ee);
    int lr = ee - 1;
    int mant = (int)(ldexp(r, -lr) * 8.0) - 8;
    return s | (uint8_t)(((lr + 7) << 3) | mant);
}

/* MX scale of one block: the smallest power of two 2^X with amax / 2^X <= 448
 * (E4M3's largest finite value), so no element of the block saturates.
 * Writing amax = m * 2^E with m in [1, 2): X = E - 8 if m <= 1.75, else
 * E - 7.  X is clamped to the UE8M0 range [-127, 127]; stored byte =
 * X + 127; amax = 0 gives byte 0.  (This rounds the scale up, as
 * TransformerEngine's MXFP8 quantiser does; the OCP v1.0 example rule
 * floor(log2 amax) - 8 would clip block maxima by up to 12.5%.) */
static int mx_scale_exp(double amax)
{
    if (amax == 0.0) return -127;
    int e;
    double m = 2.0 * frexp(amax, &e);   /* amax = m * 2^(e-1), m in [1, 2) */
    int X = (e - 1) - 8 + (m > 1.75 ? 1 : 0);
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    return X;
}

/* Quantise n_vec vectors of length K (K % 32 == 0) to MXFP8 along K.
 * Element i of vector v is in[v*stride_vec + i*stride_k] (bf16 bits).
 * Output data is K-contiguous: data[v*K + i]; scales scale[v*(K/32) + b]. */
void oracle_quantize_mxfp8(const uint16_t *in, int64_t n_vec, int64_t K,
                           int64_t stride_vec, int64_t stride_k,
                           uint8_t *data, uint8_t *scale)
{
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < n_vec; ++v) {
        for (int64_t b = 0; b < nb; ++b) {
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs(oracle_bf16_to_double(in[v * stride_vec + (b * 32 + i) * stride_k]));
                if (a > amax) amax = a;
            }
            int X = mx_scale_exp(amax);
            scale[v * nb + b] = (uint8_t)(X + 127);
            for (int i = 0; i < 32; ++i) {
                double val = oracle_bf16_to_double(in[v * stride_vec + (b * 32 + i) * stride_k]);
                data[v * K + b * 32 + i] = oracle_double_to_e4m3(ldexp(val, -X));
            }
        }
    }
}

/* Exported form of mx_fake_quant for n vectors of length K (in place allowed). */
static void mx_fake_quant(const double *in, int64_t K, double *out);
void oracle_mx_fake_quant(const double *in, int64_t n, int64_t K, double *out)
{
    for (int64_t i = 0; i < n; ++i) mx_fake_quant(in + i * K, K, out + i * K);
}

/* Same rule applied to a double vector (used for h on the MXFP8 path);
 * writes the dequantised values back to out[]. */
static void mx_fake_quant(const double *in, int64_t K, double *out)
{
    for (int64_t b = 0; b < K / 32; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            double a = fabs(in[b * 32 + i]);
            if (a > amax) amax = a;
        }
        int X = mx_scale_exp(amax);
        for (int i = 0; i < 32; ++i)
            out[b * 32 + i] = ldexp(oracle_e4m3_to_double(oracle_double_to_e4m3(ldexp(in[b * 32 + i], -X))), X);
    }
}

/* ------------------------------------------------------------------ */
/* A1: top-k routing                                                    */
/* ------------------------------------------------------------------ */

/* Ordering of (logit, expert): larger logit first; equal logits (+0 == -0)
 * go to the lower expert id; NaN ranks below every number, -inf included. */
static int ranks_before(float a, int ia, float b, int ib)
{
    int na = isnan(a), nb = isnan(b);
    if (na || nb) {
        if (na && nb) return ia < ib;
        return nb;
    }
    if (a != b) return a > b;
    return ia < ib;
}

/* For each token: the k experts first in the order above, in that order,
 * and weights w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k
 * selected logits (softmax over the selected k), computed in double and
 * rounded to fp32.  If l_0 = -inf every weight is 0. */
void oracle_route_topk(const float *logits, int64_t T, int E, int k,
                       int32_t *topk_idx, float *topk_w)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
        double lj[64];
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            taken[best] = 1;
            topk_idx[t * k + j] = best;
            lj[j] = (double)l[best];
        }
        free(taken);
        if (isinf(lj[0]) && lj[0] < 0) {
            for (int j = 0; j < k; ++j) topk_w[t * k + j] = 0.0f;
            continue;
        }
        double s = 0.0, ex[64];
        for (int j = 0; j < k; ++j) { ex[j] = exp(lj[j] - lj[0]); s += ex[j]; }
        for (int j = 0; j < k; ++j) topk_w[t * k + j] = (float)(ex[j] / s);
    }
}

/* ------------------------------------------------------------------ */
/* Router variant: sigmoid scores with an expert routing bias            */
/* ------------------------------------------------------------------ */

static double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Sigmoid score function of the fused top-k router ("[JAX] Expert
 * Parallelism: JAX primitives + VJPs", commit log: sigmoid scores, the
 * expert routing bias of the sigmoid-bias configurations, and the kernel's
 * normalisation weights / (sum + 1e-20)).  Readings: the score of expert e
 * is s_e = sigmoid(l_e); the bias takes part in the selection only (key
 * s_e + b_e, larger first, equal keys to the lower id); the weights are the
 * unbiased scores of the selected experts, divided by (their sum + 1e-20)
 * when normalize != 0.  bias may be NULL (all zero).  A NaN logit ranks
 * last.  Keys and weights in double. */
void oracle_route_topk_sigmoid(const float *logits, const float *bias, int64_t T, int E, int k,
                               int normalize, int32_t *topk_idx, float *topk_w)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        double *key = (double *)malloc((size_t)E * sizeof(double));
        unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
        for (int e = 0; e < E; ++e)
            key[e] = isnan(l[e]) ? NAN : sigmoid_d((double)l[e]) + (bias ? (double)bias[e] : 0.0);
        double s[64], sum = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0) { best = e; continue; }
                int nb = isnan(key[best]), ne = isnan(key[e]);
                if (nb && !ne) best = e;
                else if (!nb && !ne && key[e] > key[best]) best = e;
            }
            taken[best] = 1;
            topk_idx[t * k + j] = best;
            s[j] = isnan(l[best]) ? 0.0 : sigmoid_d((double)l[best]);
            sum += s[j];
        }
        for (int j = 0; j < k; ++j)
            topk_w[t * k + j] = (float)(normalize ? s[j] / (sum + 1e-20) : s[j]);
        free(taken);
        free(key);
    }
}

/* Router backward: d_logits [T, E] (double) from d_topk_w [T, k] for the
 * selection topk_idx (ids outside [0, E) are skipped), following the router's
 * VJP ("[JAX] Expert Parallelism: JAX primitives + VJPs", commit log:
 * fused_topk_with_score_function_bwd produces the fp32 logits cotangent).
 * The weights are recomputed in double from the logits; unselected experts
 * get 0 (the selection is piecewise constant), and so does the bias.
 *   score_fn 0 (softmax over the k selected):  dl_j = w_j (g_j - sum_i w_i g_i)
 *   score_fn 1 (sigmoid s_j):  normalize: ds_j = (g_j - sum_i w_i g_i) / (S + 1e-20),
 *                              else ds_j = g_j;  dl_j = ds_j s_j (1 - s_j)      */
void oracle_route_topk_bwd(const float *logits, const int32_t *topk_idx, const float *d_topk_w,
                           int64_t T, int E, int k, int score_fn, int normalize, double *d_logits)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        double *dl = d_logits + t * E;
        for (int e = 0; e < E; ++e) dl[e] = 0.0;
        double w[64], s[64], g[64];
        int id[64], n = 0;
        for (int j = 0; j < k; ++j) {
            int e = topk_idx[t * k + j];
            if (e < 0 || e >= E) continue;
            id[n] = e;
            g[n] = (double)d_topk_w[t * k + j];
            ++n;
        }
        if (n == 0) continue;
        if (score_fn == 0) {
            double lmax = -INFINITY, sum = 0.0;
            for (int j = 0; j < n; ++j)
                if ((double)l[id[j]] > lmax) lmax = (double)l[id[j]];
            if (isinf(lmax) && lmax < 0) continue;   /* all weights 0, no gradient */
            for (int j = 0; j < n; ++j) { w[j] = exp((double)l[id[j]] - lmax); sum += w[j]; }
            double gw = 0.0;
            for (int j = 0; j < n; ++j) { w[j] /= sum; gw += w[j] * g[j]; }
            for (int j = 0; j < n; ++j) dl[id[j]] += w[j] * (g[j] - gw);
        } else {
            double S = 0.0;
            for (int j = 0; j < n; ++j) { s[j] = sigmoid_d((double)l[id[j]]); S += s[j]; }
            double gw = 0.0;
            if (normalize)
                for (int j = 0; j < n; ++j) gw += g[j] * s[j] / (S + 1e-20);
            for (int j = 0; j < n; ++j) {
                double ds = normalize ? (g[j] - gw) / (S + 1e-20) : g[j];
                dl[id[j]] += ds * s[j] * (1.0 - s[j]);
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* A2: permutation into expert-contiguous order                         */
/* ------------------------------------------------------------------ */

/* Routes are flattened r = t*k + j.  group_sizes[e] = #{r : idx[r] == e};
 * each group occupies round_up(size, align) rows starting at
 * group_offsets[e] (exclusive prefix sum); group_offsets[E] = rows used.
 * Within a group rows follow ascending r (a stable counting sort).
 * dst_of_route[r] = row of route r, -1 for a dropped (-1) or invalid route;
 * src_of_row[row] = r, -1 for a padding row.  Ids outside [-1, E) count as
 * errors and are dropped.  Returns the number of invalid ids. */
int64_t oracle_permute(const int32_t *topk_idx, int64_t T, int k, int E, int align,
                       int32_t *dst_of_route, int32_t *src_of_row, int64_t rows_cap,
                       int32_t *group_sizes, int32_t *group_offsets)
{
    int64_t R = T * k, bad = 0;
    for (int e = 0; e < E; ++e) group_sizes[e] = 0;
    for (int64_t r = 0; r < R; ++r) {
        int32_t e = topk_idx[r];
        if (e >= 0 && e < E) group_sizes[e]++;
        else if (e != -1) bad++;
    }
    group_offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        int64_t padded = ((int64_t)group_sizes[e] + align - 1) / align * align;
        group_offsets[e + 1] = (int32_t)(group_offsets[e] + padded);
    }
    for (int64_t i = 0; i < rows_cap; ++i) src_of_row[i] = -1;
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t r = 0; r < R; ++r) {
        int32_t e = topk_idx[r];
        if (e >= 0 && e < E) {
            int32_t row = group_offsets[e] + fill[e]++;
            dst_of_route[r] = row;
            src_of_row[row] = (int32_t)r;
        } else {
            dst_of_route[r] = -1;
        }
    }
    free(fill);
    return bad;
}

/* x_perm[row] = x[src_of_row[row] / k], zero for padding rows (bf16 bits). */
void oracle_gather_rows(const uint16_t *x, int H, int k, const int32_t *src_of_row,
                        int64_t rows, uint16_t *x_perm)
{
    for (int64_t i = 0; i < rows; ++i) {
        if (src_of_row[i] < 0) memset(x_perm + i * H, 0, (size_t)H * 2);
        else memcpy(x_perm + i * H, x + (int64_t)(src_of_row[i] / k) * H, (size_t)H * 2);
    }
}

/* A5 on its own: out[t] = sum_j w[t,j] * y_perm[dst_of_route[t,j]] in slot
 * order, dropped routes (-1) skipped (double; bf16 in round_mode 1). */
void oracle_unpermute_combine(const float *y_perm, const int32_t *dst_of_route,
                              const float *topk_w, int64_t T, int H, int k,
                              int round_mode, double *out)
{
    for (int64_t t = 0; t < T; ++t) {
        double *o = out + t * H;
        for (int n = 0; n < H; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int32_t row = dst_of_route[t * k + j];
            if (row < 0) continue;
            double w = (double)topk_w[t * k + j];
            for (int n = 0; n < H; ++n) o[n] += w * (double)y_perm[(int64_t)row * H + n];
        }
        for (int n = 0; n < H; ++n) o[n] = rnd_out(o[n], round_mode);
    }
}

/* The combine with an MXFP8 output encoding ("Add MoE + expert-parallel Python API
 * surface, PyTorch reference, and tests", Summary: bf16, mxfp8 and nvfp4 public
 * outputs as block-scaled tensors in their logical, unswizzled layout).  The sum is
 * the combine's own: fp32, slot order, one rounding per multiply-add (fmaf), dropped
 * routes skipped, starting from +0; its fp32 value then takes the MX rule along H:
 * codes [T, H] (E4M3) and scales [T, H/32] (UE8M0, row-major).  The codes are
 * decided on the fp32 value, as the kernel decides them. */
void oracle_unpermute_combine_mxfp8(const float *y_perm, const int32_t *dst_of_route,
                                    const float *topk_w, int64_t T, int H, int k,
                                    uint8_t *codes, uint8_t *scales)
{
    float *acc = (float *)malloc(sizeof(float) * (size_t)H);
    for (int64_t t = 0; t < T; ++t) {
        for (int n = 0; n < H; ++n) acc[n] = 0.0f;
        for (int j = 0; j < k; ++j) {
            int32_t row = dst_of_route[t * k + j];
            if (row < 0) continue;
            const float w = topk_w[t * k + j];
            for (int n = 0; n < H; ++n) acc[n] = fmaf(w, y_perm[(int64_t)row * H + n], acc[n]);
        }
        for (int b = 0; b < H / 32; ++b) {
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs((double)acc[b * 32 + i]);
                if (a > amax) amax = a;
            }
            int X = mx_scale_exp(amax);
            scales[t * (H / 32) + b] = (uint8_t)(X + 127);
            for (int i = 0; i < 32; ++i)
                codes[t * H + b * 32 + i] = oracle_double_to_e4m3(ldexp((double)acc[b * 32 + i], -X));
        }
    }
    free(acc);
}

/* The combine with an NVFP4 output encoding ("Add MoE + expert-parallel Python API
 * surface, PyTorch reference, and tests", Summary: nvfp4 public outputs as block-scaled
 * tensors in their logical layout; BlockScaledTensor: data plus one scale per block,
 * block_size 16 for nvfp4, and no tensor-level scale in the bundle).  The pages fix
 * neither the element nor the scale format beyond that; the reading taken here:
 *   elements: FP4 E2M1 (sign, 2 exponent bits, 1 mantissa bit), magnitudes
 *             0, 0.5, 1, 1.5, 2, 3, 4, 6, in blocks of 16 consecutive elements along H;
 *   scale:    one FP8 E4M3 value s per block, the smallest positive finite E4M3 value
 *             with 6 s >= amax (so no element clips); 448 when amax > 6 * 448 (those
 *             elements saturate at 6 s); byte 0x00 (s = 0, every code 0) when amax = 0;
 *   codes:    the E2M1 magnitude nearest to |v| / s, a tie going to the magnitude whose
 *             mantissa bit is 0; sign bit set when v < 0; two codes per byte, element
 *             2i in the low nibble.
 * Decoded value: (-1)^sign * magnitude * s.  The sum is the combine's own fp32
 * slot-order sum (fmaf, from +0, dropped routes skipped), as for the MXFP8 output.
 * codes [T, H/2], scales [T, H/16] (E4M3 bytes, row-major). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* smallest E4M3 code in [1, 0x7E] whose value s has 6 s >= amax; 0 for amax = 0 */
static uint8_t nvfp4_scale_code(double amax)
{
    if (amax == 0.0) return 0;
    for (int c = 1; c <= 0x7E; ++c)
        if (6.0 * oracle_e4m3_to_double((uint8_t)c) >= amax) return (uint8_t)c;
    return 0x7E;
}

/* 4-bit code of v at block scale s > 0: nearest magnitude, ties to the even index */
static uint8_t nvfp4_code(double v, double s)
{
    const double a = fabs(v);
    int best = 0;
    double bd = a;
    for (int m = 1; m < 8; ++m) {
        const double d = fabs(a - s * E2M1_MAG[m]);
        if (d < bd || (d == bd && (m & 1) == 0)) { bd = d; best = m; }
    }
    return (uint8_t)((v < 0 ? 8 : 0) | best);
}

void oracle_nvfp4_encode(const float *v, int64_t n_blocks, uint8_t *codes, uint8_t *scales)
{
    for (int64_t b = 0; b < n_blocks; ++b) {
        double amax = 0.0;
        for (int i = 0; i < 16; ++i) {
            double a = fabs((double)v[b * 16 + i]);
            if (a > amax) amax = a;
        }
        const uint8_t sc = nvfp4_scale_code(amax);
        scales[b] = sc;
        const double s = oracle_e4m3_to_double(sc);
        for (int i = 0; i < 8; ++i) {
            uint8_t lo = 0, hi = 0;
            if (sc) {
                lo = nvfp4_code((double)v[b * 16 + 2 * i], s);
                hi = nvfp4_code((double)v[b * 16 + 2 * i + 1], s);
            }
            codes[b * 8 + i] = (uint8_t)(lo | (hi << 4));
        }
    }
}

double oracle_nvfp4_value(uint8_t code, uint8_t scale)
{
    const double m = E2M1_MAG[code & 7] * oracle_e4m3_to_double(scale);
    return (code & 8) ? -m : m;
}

void oracle_unpermute_combine_nvfp4(const float *y_perm, const int32_t *dst_of_route,
                                    const float *topk_w, int64_t T, int H, int k,
                                    uint8_t *codes, uint8_t *scales)
{
    float *acc = (float *)malloc(sizeof(float) * (size_t)H);
    for (int64_t t = 0; t < T; ++t) {
        for (int n = 0; n < H; ++n) acc[n] = 0.0f;
        for (int j = 0; j < k; ++j) {
            int32_t row = dst_of_route[t * k + j];
            if (row < 0) continue;
            const float w = topk_w[t * k + j];
            for (int n = 0; n < H; ++n) acc[n] = fmaf(w, y_perm[(int64_t)row * H + n], acc[n]);
        }
        oracle_nvfp4_encode(acc, H / 16, codes + t * (H / 2), scales + t * (H / 16));
    }
    free(acc);
}

/* ------------------------------------------------------------------ */
/* A3/A4: one route through one expert                                  */
/* ------------------------------------------------------------------ */

static double silu(double g) { return g / (1.0 + exp(-g)); }
static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

/* Optional clamp of the SwiGLU inputs ("Add MoE + expert-parallel Python API surface,
 * PyTorch reference, and tests", Summary: local SwiGLU experts with an optional
 * DeepSeek-style clamp; inclusive clamp bounds).  The pages give no form and no
 * values; reading: the gate and up accumulators are clamped to caller-given
 * intervals before SwiGLU, h = silu(clamp(g, gate_lo, gate_hi)) * clamp(u, up_lo,
 * up_hi), and "inclusive" means a value equal to a bound is inside: its derivative
 * passes, a value outside gets derivative 0.  +-inf bounds (the default) disable it.
 * Set for the whole library (before any parallel region runs). */
static double g_gate_lo = -INFINITY, g_gate_hi = INFINITY, g_up_lo = -INFINITY, g_up_hi = INFINITY;

void oracle_set_swiglu_clamp(double gate_lo, double gate_hi, double up_lo, double up_hi)
{
    g_gate_lo = gate_lo; g_gate_hi = gate_hi; g_up_lo = up_lo; g_up_hi = up_hi;
}

static double clamp_to(double v, double lo, double hi) { return v < lo ? lo : (v > hi ? hi : v); }
static double inside(double v, double lo, double hi) { return (v >= lo && v <= hi) ? 1.0 : 0.0; }
static double swiglu(double g, double u)
{
    return silu(clamp_to(g, g_gate_lo, g_gate_hi)) * clamp_to(u, g_up_lo, g_up_hi);
}

/* One route through one expert: g = x Wg, u = x Wu (double), h = rnd(hw * silu(g) * u)
 * and y = rnd(yw * (h Wd)), both stored bf16 on the path (rounded in round_mode 1
 * and 2).  hw = w when the router weight is applied in the FC1 epilogue, yw = w when
 * it is applied in the FC2 epilogue (the fp32 product is what the path rounds), else
 * 1.  h_mx != 0: the MXFP8 forward's h instead, hw * silu(g) * u quantised to MXFP8
 * along F and dequantised (in every round mode: the quantisation is part of that
 * forward).  Wg, Wu are [H,F]; Wd is [F,H]. */
static void expert_route(const uint16_t *xr, const uint16_t *Wg, const uint16_t *Wu,
                         const uint16_t *Wd, int H, int F, int round_mode, double hw, double yw, int h_mx,
                         double *g, double *u, double *h, double *y)
{
    for (int f = 0; f < F; ++f) { g[f] = 0.0; u[f] = 0.0; }
    for (int i = 0; i < H; ++i) {
        double xv = oracle_bf16_to_double(xr[i]);
        const uint16_t *wg = Wg + (int64_t)i * F, *wu = Wu + (int64_t)i * F;
        for (int f = 0; f < F; ++f) {
            g[f] += xv * oracle_bf16_to_double(wg[f]);
            u[f] += xv * oracle_bf16_to_double(wu[f]);
        }
    }
    if (h_mx) {
        for (int f = 0; f < F; ++f) h[f] = hw * swiglu(g[f], u[f]);
        mx_fake_quant(h, F, h);
    } else {
        for (int f = 0; f < F; ++f) h[f] = rnd(hw * swiglu(g[f], u[f]), round_mode);
    }
    for (int n = 0; n < H; ++n) y[n] = 0.0;
    for (int f = 0; f < F; ++f) {
        const uint16_t *wd = Wd + (int64_t)f * H;
        for (int n = 0; n < H; ++n) y[n] += h[f] * oracle_bf16_to_double(wd[n]);
    }
    for (int n = 0; n < H; ++n) y[n] = rnd(yw * y[n], round_mode);
}

/* ------------------------------------------------------------------ */
/* Forward (A1..A5) for a list of tokens                                */
/* ------------------------------------------------------------------ */

/* out[i] (double [n_tokens, H]) = sum_j w[t,j] * y(t,j) for t = tokens[i]
 * (all tokens when tokens == NULL), slot order, dropped routes skipped,
 * rounded to bf16 in round_mode 1.  Optional per-route outputs, indexed
 * [i*k + j]: fc1 (double [.., 2F], g then u, unrounded), h [.., F], y [.., H];
 * rows of dropped routes are left untouched.  Weights are given per expert
 * (Wg[e], Wu[e]: [H,F]; Wd[e]: [F,H]); only routed experts are read. */
/* Where the router weight w of a route is applied ("Add MoE + expert-parallel Python
 * API surface, PyTorch reference, and tests", Summary: the router weight in the FC1 or
 * FC2 epilogue; "[JAX] Expert Parallelism", commit log: apply_topk_weights_early):
 *   weight_at 0  in the combine: out = sum_j w_j y_j            (late, the default)
 *   weight_at 1  in FC1:  h_j = rnd(w_j silu(g) u), out = sum_j y_j
 *   weight_at 2  in FC2:  y_j = rnd(w_j (h_j Wd)),  out = sum_j y_j
 * All three are the same function in exact arithmetic; they differ in where the
 * roundings of h and y fall (weight_at 1 rounds the weighted h, weight_at 2 the
 * weighted y).  y_out holds the per-route y as the path stores it (weighted for 1
 * and 2). */
void oracle_moe_fwd_w(int64_t n_tokens, const int64_t *tokens, int H, int F, int E, int k,
                      const uint16_t *x, const uint16_t *const *Wg, const uint16_t *const *Wu,
                      const uint16_t *const *Wd, const int32_t *topk_idx, const float *topk_w,
                      int round_mode, int weight_at, int h_mx, double *out, double *fc1, double *h_out,
                      double *y_out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        double *g = (double *)malloc(sizeof(double) * (size_t)(3 * F + H));
        double *u = g + F, *h = u + F, *y = h + F;
        double *o = out + i * H;
        for (int n = 0; n < H; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int32_t e = topk_idx[t * k + j];
            if (e < 0 || e >= E) continue;
            const double w = (double)topk_w[t * k + j];
            expert_route(x + t * H, Wg[e], Wu[e], Wd[e], H, F, round_mode, weight_at == 1 ? w : 1.0,
                         weight_at == 2 ? w : 1.0, h_mx, g, u, h, y);
            const double wc = weight_at == 0 ? w : 1.0;
            for (int n = 0; n < H; ++n) o[n] += wc * y[n];
            int64_t ri = i * k + j;
            if (fc1) { memcpy(fc1 + ri * 2 * F, g, sizeof(double) * F); memcpy(fc1 + ri * 2 * F + F, u, sizeof(double) * F); }
            if (h_out) memcpy(h_out + ri * F, h, sizeof(double) * F);
            if (y_out) memcpy(y_out + ri * H, y, sizeof(double) * H);
        }
        for (int n = 0; n < H; ++n) o[n] = rnd_out(o[n], round_mode);
        free(g);
    }
}

void oracle_moe_fwd(int64_t n_tokens, const int64_t *tokens, int H, int F, int E, int k,
                    const uint16_t *x, const uint16_t *const *Wg, const uint16_t *const *Wu,
                    const uint16_t *const *Wd, const int32_t *topk_idx, const float *topk_w,
                    int round_mode, double *out, double *fc1, double *h_out, double *y_out)
{
    oracle_moe_fwd_w(n_tokens, tokens, H, F, E, k, x, Wg, Wu, Wd, topk_idx, topk_w, round_mode, 0, 0, out, fc1,
                     h_out, y_out);
}

/* ------------------------------------------------------------------ */
/* A7: MXFP8 forward for a list of tokens                               */
/* ------------------------------------------------------------------ */

/* As oracle_moe_fwd, but every GEMM operand is MXFP8 (E4M3 + UE8M0 per 1x32
 * block along K) and dequantised exactly: x along H; W_gate / W_up given as
 * quantised K-major [F][H] codes with scales [F][H/32]; W_down as quantised
 * [H][F] codes with scales [H][F/32]; h = silu(g)*u quantised along F from
 * its unrounded value.  y is stored bf16 (rounded in round_mode 1 and 2); out
 * is bf16 in round_mode 1. */
void oracle_moe_fwd_mxfp8(int64_t n_tokens, const int64_t *tokens, int H, int F, int E, int k,
                          const uint16_t *x,
                          const uint8_t *const *Wg_q, const uint8_t *const *Wg_s,
                          const uint8_t *const *Wu_q, const uint8_t *const *Wu_s,
                          const uint8_t *const *Wd_q, const uint8_t *const *Wd_s,
                          const int32_t *topk_idx, const float *topk_w, int round_mode,
                          double *out, double *y_out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        double *xd = (double *)malloc(sizeof(double) * (size_t)(2 * H + 3 * F));
        double *y = xd + H, *g = y + H, *u = g + F, *h = u + F;
        uint8_t *xq = (uint8_t *)malloc((size_t)H + (size_t)H / 32);
        uint8_t *xs = xq + H;
        oracle_quantize_mxfp8(x + t * H, 1, H, H, 1, xq, xs);
        for (int n = 0; n < H; ++n) xd[n] = ldexp(oracle_e4m3_to_double(xq[n]), (int)xs[n / 32] - 127);
        double *o = out + i * H;
        for (int n = 0; n < H; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int32_t e = topk_idx[t * k + j];
            if (e < 0 || e >= E) continue;
            for (int f = 0; f < F; ++f) {
                double sg = 0.0, su = 0.0;
                const uint8_t *qg = Wg_q[e] + (int64_t)f * H, *qu = Wu_q[e] + (int64_t)f * H;
                const uint8_t *cg = Wg_s[e] + (int64_t)f * (H / 32), *cu = Wu_s[e] + (int64_t)f * (H / 32);
                for (int n = 0; n < H; ++n) {
                    sg += xd[n] * ldexp(oracle_e4m3_to_double(qg[n]), (int)cg[n / 32] - 127);
                    su += xd[n] * ldexp(oracle_e4m3_to_double(qu[n]), (int)cu[n / 32] - 127);
                }
                g[f] = sg;
                u[f] = su;
                h[f] = swiglu(sg, su);
            }
            mx_fake_quant(h, F, h);
            for (int n = 0; n < H; ++n) {
                double s = 0.0;
                const uint8_t *qd = Wd_q[e] + (int64_t)n * F, *cd = Wd_s[e] + (int64_t)n * (F / 32);
                for (int f = 0; f < F; ++f) s += h[f] * ldexp(oracle_e4m3_to_double(qd[f]), (int)cd[f / 32] - 127);
                y[n] = rnd(s, round_mode);
            }
            double w = (double)topk_w[t * k + j];
            for (int n = 0; n < H; ++n) o[n] += w * y[n];
            if (y_out) memcpy(y_out + (i * k + j) * H, y, sizeof(double) * H);
        }
        for (int n = 0; n < H; ++n) o[n] = rnd_out(o[n], round_mode);
        free(xq);
        free(xd);
    }
}

/* ------------------------------------------------------------------ */
/* A8: backward                                                         */
/* ------------------------------------------------------------------ */

/* Per-route backward pieces for route (t, j) -> e, given dY[t]:
 *   dy    = w * dY[t]                               (bf16 in round_mode 1)
 *   dh    = dy Wd^T                                 (length F)
 *   with G, U = the fc1_c stash (bf16 of g, u) in round_mode 1, else g, u:
 *   dg    = dh * U * s * (1 + G * (1 - s)),  s = sigmoid(G)   (bf16 in mode 1)
 *   du    = dh * G * s                                      (bf16 in mode 1)
 *   dxr   = dg Wg^T + du Wu^T                       (unrounded: fp32 on the path)
 * g, u, h are the forward values of the route. */
static void route_bwd(const uint16_t *dYt, double w, const double *g, const double *u,
                      const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd,
                      int H, int F, int round_mode,
                      double *dy, double *dg, double *du, double *dxr)
{
    for (int n = 0; n < H; ++n) dy[n] = rnd(w * oracle_bf16_to_double(dYt[n]), round_mode);
    for (int f = 0; f < F; ++f) {
        const uint16_t *wd = Wd + (int64_t)f * H;
        double dh = 0.0;
        for (int n = 0; n < H; ++n) dh += dy[n] * oracle_bf16_to_double(wd[n]);
        double G = rnd(g[f], round_mode), U = rnd(u[f], round_mode);
        double Gc = clamp_to(G, g_gate_lo, g_gate_hi), Uc = clamp_to(U, g_up_lo, g_up_hi);
        double s = sigmoid(Gc);
        dg[f] = rnd(inside(G, g_gate_lo, g_gate_hi) * dh * Uc * s * (1.0 + Gc * (1.0 - s)), round_mode);
        du[f] = rnd(inside(U, g_up_lo, g_up_hi) * dh * Gc * s, round_mode);
    }
    if (!dxr) return;
    for (int i = 0; i < H; ++i) {
        const uint16_t *wg = Wg + (int64_t)i * F, *wu = Wu + (int64_t)i * F;
        double s = 0.0;
        for (int f = 0; f < F; ++f)
            s += dg[f] * oracle_bf16_to_double(wg[f]) + du[f] * oracle_bf16_to_double(wu[f]);
        dxr[i] = s;
    }
}

/* Full backward (small problems).  Inputs as oracle_moe_fwd plus dY bf16
 * [T,H].  Outputs (double): dx [T,H] = sum_j dxr(t,j) (bf16 in mode 1);
 * dWg, dWu [E,H,F] = sum over routes of x^T dg / x^T du; dWd [E,F,H] = sum
 * over routes of h^T dy (each bf16 in mode 1); experts with no route get
 * exactly 0.  d_topk_w [T,k] = <dY[t], y(t,j)> with y as the forward stores it
 * (bf16 in round_mode 1 and 2; 0 for dropped routes).
 *
 * h_mx != 0: the straight-through backward of the MXFP8 forward ("Add MoE +
 * expert-parallel Python API surface, PyTorch reference, and tests", Summary:
 * quantization round-trips are straight-through).  x and the weights are then
 * passed as their MXFP8 round trips (bf16 bit patterns of the dequantised
 * values), h is the forward's MXFP8 h (expert_route), and every derivative
 * treats a quantisation as the identity: the formulas above are unchanged. */
void oracle_moe_bwd(int64_t T, int H, int F, int E, int k, const uint16_t *x,
                    const uint16_t *const *Wg, const uint16_t *const *Wu, const uint16_t *const *Wd,
                    const int32_t *topk_idx, const float *topk_w, const uint16_t *dY,
                    int round_mode, int h_mx, double *dx, double *dWg, double *dWu, double *dWd,
                    double *d_topk_w)
{
    memset(dWg, 0, sizeof(double) * (size_t)E * H * F);
    memset(dWu, 0, sizeof(double) * (size_t)E * H * F);
    memset(dWd, 0, sizeof(double) * (size_t)E * F * H);
    double *g = (double *)malloc(sizeof(double) * (size_t)(6 * F + 4 * H));
    double *u = g + F, *h = u + F, *dg = h + F, *du = dg + F, *unused = du + F;
    double *y = unused + F, *dy = y + H, *dxr = dy + H, *acc = dxr + H;
    for (int64_t t = 0; t < T; ++t) {
        for (int n = 0; n < H; ++n) acc[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int32_t e = topk_idx[t * k + j];
            if (e < 0 || e >= E) { d_topk_w[t * k + j] = 0.0; continue; }
            expert_route(x + t * H, Wg[e], Wu[e], Wd[e], H, F, round_mode, 1.0, 1.0, h_mx, g, u, h, y);
            double dw = 0.0;
            for (int n = 0; n < H; ++n) dw += oracle_bf16_to_double(dY[t * H + n]) * y[n];
            d_topk_w[t * k + j] = dw;
            route_bwd(dY + t * H, (double)topk_w[t * k + j], g, u, Wg[e], Wu[e], Wd[e], H, F,
                      round_mode, dy, dg, du, dxr);
            for (int n = 0; n < H; ++n) acc[n] += dxr[n];
            double *wg = dWg + (int64_t)e * H * F, *wu = dWu + (int64_t)e * H * F, *wd = dWd + (int64_t)e * F * H;
            for (int i = 0; i < H; ++i) {
                double xv = oracle_bf16_to_double(x[t * H + i]);
                for (int f = 0; f < F; ++f) {
                    wg[(int64_t)i * F + f] += xv * dg[f];
                    wu[(int64_t)i * F + f] += xv * du[f];
                }
            }
            for (int f = 0; f < F; ++f)
                for (int n = 0; n < H; ++n) wd[(int64_t)f * H + n] += h[f] * dy[n];
        }
        for (int n = 0; n < H; ++n) dx[t * H + n] = rnd_out(acc[n], round_mode);
    }
    free(g);
    /* the weight gradients are fp32 on the path: no bf16 rounding in any mode */
}

/* dx and d_topk_w for a list of tokens (any problem size): dx[i] (double
 * [n_tokens, H]) and d_topk_w[i*k + j], as in oracle_moe_bwd (h_mx likewise). */
void oracle_moe_bwd_dx_tokens(int64_t n_tokens, const int64_t *tokens, int H, int F, int E, int k,
                              const uint16_t *x, const uint16_t *const *Wg, const uint16_t *const *Wu,
                              const uint16_t *const *Wd, const int32_t *topk_idx, const float *topk_w,
                              const uint16_t *dY, int round_mode, int h_mx, double *dx, double *d_topk_w)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        double *g = (double *)malloc(sizeof(double) * (size_t)(5 * F + 3 * H));
        double *u = g + F, *h = u + F, *dg = h + F, *du = dg + F;
        double *y = du + F, *dy = y + H, *dxr = dy + H;
        double *o = dx + i * H;
        for (int n = 0; n < H; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int32_t e = topk_idx[t * k + j];
            if (e < 0 || e >= E) { d_topk_w[i * k + j] = 0.0; continue; }
            expert_route(x + t * H, Wg[e], Wu[e], Wd[e], H, F, round_mode, 1.0, 1.0, h_mx, g, u, h, y);
            double dw = 0.0;
            for (int n = 0; n < H; ++n) dw += oracle_bf16_to_double(dY[t * H + n]) * y[n];
            d_topk_w[i * k + j] = dw;
            route_bwd(dY + t * H, (double)topk_w[t * k + j], g, u, Wg[e], Wu[e], Wd[e], H, F,
                      round_mode, dy, dg, du, dxr);
            for (int n = 0; n < H; ++n) o[n] += dxr[n];
        }
        for (int n = 0; n < H; ++n) o[n] = rnd_out(o[n], round_mode);
        free(g);
    }
}

/* Single weight-gradient entries (any problem size).  Entry q is
 * (which[q], e[q], a[q], b[q]) with which = 0: dWg[e][a=h][b=f],
 * 1: dWu[e][a=h][b=f], 2: dWd[e][a=f][b=n].  Each is the plain sum over the
 * routes r = (t, j) with topk_idx[r] == e of x[t][h]*dg_r[f], x[t][h]*du_r[f]
 * or h_r[f]*dy_r[n], evaluated from its definition one entry at a time. */
void oracle_moe_bwd_dw_entries(int64_t n_entries, const int32_t *which, const int32_t *ent_e,
                               const int32_t *ent_a, const int32_t *ent_b,
                               int64_t T, int H, int F, int E, int k, const uint16_t *x,
                               const uint16_t *const *Wg, const uint16_t *const *Wu,
                               const uint16_t *const *Wd, const int32_t *topk_idx,
                               const float *topk_w, const uint16_t *dY, int round_mode, int h_mx,
                               double *val)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < n_entries; ++q) {
        int e = ent_e[q], wsel = which[q];
        int f = (wsel == 2) ? ent_a[q] : ent_b[q];
        int hn = (wsel == 2) ? ent_b[q] : ent_a[q];
        double acc = 0.0;
        for (int64_t r = 0; r < T * k; ++r) {
            if (topk_idx[r] != e) continue;
            int64_t t = r / k;
            const uint16_t *xr = x + t * H;
            double g = 0.0, u = 0.0;
            for (int i = 0; i < H; ++i) {
                double xv = oracle_bf16_to_double(xr[i]);
                g += xv * oracle_bf16_to_double(Wg[e][(int64_t)i * F + f]);
                u += xv * oracle_bf16_to_double(Wu[e][(int64_t)i * F + f]);
            }
            double w = (double)topk_w[r];
            if (wsel == 2) {
                double h = rnd(swiglu(g, u), round_mode);
                if (h_mx) {   /* MXFP8 h: the whole 32-wide block of f along F */
                    double hb[32];
                    const int f0 = f / 32 * 32;
                    for (int c = 0; c < 32; ++c) {
                        double gc = 0.0, uc = 0.0;
                        for (int i = 0; i < H; ++i) {
                            double xv = oracle_bf16_to_double(xr[i]);
                            gc += xv * oracle_bf16_to_double(Wg[e][(int64_t)i * F + f0 + c]);
                            uc += xv * oracle_bf16_to_double(Wu[e][(int64_t)i * F + f0 + c]);
                        }
                        hb[c] = swiglu(gc, uc);
                    }
                    mx_fake_quant(hb, 32, hb);
                    h = hb[f - f0];
                }
                double dy = rnd(w * oracle_bf16_to_double(dY[t * H + hn]), round_mode);
                acc += h * dy;
            } else {
                double dh = 0.0;
                const uint16_t *wd = Wd[e] + (int64_t)f * H;
                for (int n = 0; n < H; ++n)
                    dh += rnd(w * oracle_bf16_to_double(dY[t * H + n]), round_mode) * oracle_bf16_to_double(wd[n]);
                double G = rnd(g, round_mode), U = rnd(u, round_mode);
                double Gc = clamp_to(G, g_gate_lo, g_gate_hi), Uc = clamp_to(U, g_up_lo, g_up_hi);
                double s = sigmoid(Gc);
                double d = (wsel == 0)
                               ? rnd(inside(G, g_gate_lo, g_gate_hi) * dh * Uc * s * (1.0 + Gc * (1.0 - s)), round_mode)
                               : rnd(inside(U, g_up_lo, g_up_hi) * dh * Gc * s, round_mode);
                acc += oracle_bf16_to_double(xr[hn]) * d;
            }
        }
        val[q] = acc;   /* fp32 on the path: not rounded */
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Round n doubles to bf16 values (returned as doubles). */
void oracle_round_bf16_array(const double *in, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = bf(in[i]);
}
