/*
 * sga_oracle.c -- slow, plain, fp64 CPU oracle for Subsampling Global Attention (SGA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or calls
 * this file; only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * load it (through ctypes).  It shares no code, header, table or constant with the CUDA
 * path.  It is written for a reader to check against the pages by eye: no blocking, no
 * fusion, no reordering beyond what the method's definition states.
 *
 * Sources (web pages, cited by title and section):
 *   [AVGGT]   "AVGGT: Rethinking Global Attention for Accelerating VGGT" (CVPR 2026 notes),
 *             Key design 1 (Global-to-Frame), Key design 2 (SGA, with the standard attention
 *             equation), Key design 3 (diagonal retention + mean fill, shared softmax).
 *   [AVGGT-de] the German technical summary of the same paper, section 2.B.
 *   [Regime]  "RegimeVGGT: Layer-Wise Spatially Preserving Redundancy Removal for Visual
 *             Geometry Grounded Transformer" (NeurIPS 2026 notes), "Core mechanism"
 *             (L = T + 5 tokens per frame), Key design 2 (size-aware attention
 *             softmax(QK^T/sqrt(d) + log g^T) V), Key design 3 (phase-shifted grid,
 *             frame-0 anchor, camera/register tokens at full density).
 *
 * Readings taken where the pages are silent (each is a parameter or a documented rule):
 *   R1  the n_special camera/register tokens occupy the first slots p = 0..n_special-1 of a
 *       frame; patches follow in row-major order, p = n_special + r*grid_w + c.
 *   R2  "first token of each s_h x s_w window": windows tile the grid from (0,0); a partial
 *       edge window keeps its top-left token.  Equivalently r % s_h == 0 && c % s_w == 0.
 *   R3  phase shift for a (s_h, s_w) grid: row offset (f div s_w) mod s_h, column offset
 *       f mod s_w (the RegimeVGGT formula with tile t, generalised per axis); a kept patch
 *       satisfies r == phi_r (mod s_h) and c == phi_c (mod s_w).  f is the global frame index.
 *   R4  the diagonal term exists only for a query whose own token was dropped (a kept
 *       query already sees itself through S; the three components are disjoint).
 *   R5  mean term, leave-one-out (default): for a dropped query i the mean runs over
 *       D \ {i} with count c-1; for a kept query over D with count c.  mean_mode = 1 selects
 *       the plain global mean over D with count c for every query.
 *   R6  the size-aware bias is + ln(count) added after the 1/sqrt(d) scaling; no mean term
 *       when its count is 0.
 *   R7  the mean is per (batch, head) over every dropped token of every frame.
 *
 * Parity pins (in tests/): closed-form kept counts; the page's sigma map and phase formula;
 * sigma = 1 equals textbook attention and torch SDPA in fp64; the frame variant equals
 * per-frame attention; with all dropped keys/values equal the SGA output equals dense
 * attention exactly; Q = 0 gives the mean of all values; an explicit per-query brute force
 * agrees.  The semantic readings R1, R3 (non-square), R4 and R5 themselves cannot be
 * pinned by the pages: parity unpinned for those choices beyond the invariants above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------------------
 * Plan: the kept key/value set S.  [AVGGT] Key design 2; [Regime] Key design 3.
 * Direct double loop over frames f and in-frame slots p.  Writes
 *   kept[t]      1 if token t = f*L + p is a key/value of S, else 0   (T entries)
 *   kv_index[s]  the tokens of S in ascending order                    (capacity T)
 *   frame_off[f] index into kv_index of frame f's first kept token     (N+1 entries)
 * Returns |S|, or -1 on a bad argument.
 * ------------------------------------------------------------------------------------ */
int64_t oracle_plan(int N, int grid_h, int grid_w, int n_special, int s_h, int s_w,
                    int phase_shift, int ref_frame_dense,
                    uint8_t* kept, int32_t* kv_index, int32_t* frame_off)
{
    if (N <= 0 || grid_h <= 0 || grid_w <= 0 || n_special < 0 || s_h <= 0 || s_w <= 0)
        return -1;
    const int64_t L = (int64_t)n_special + (int64_t)grid_h * grid_w;
    int64_t n_kept = 0;
    for (int f = 0; f < N; ++f) {
        frame_off[f] = (int32_t)n_kept;
        int phi_r = 0, phi_c = 0;
        if (phase_shift) {
            phi_r = (f / s_w) % s_h;
            phi_c = f % s_w;
        }
        for (int64_t p = 0; p < L; ++p) {
            const int64_t t = (int64_t)f * L + p;
            int keep = 0;
            if (f == 0 && ref_frame_dense) {
                keep = 1;                       /* reference frame uncompressed */
            } else if (p < n_special) {
                keep = 1;                       /* camera / register tokens at full density */
            } else {
                const int64_t r = (p - n_special) / grid_w;
                const int64_t c = (p - n_special) % grid_w;
                if (r % s_h == phi_r && c % s_w == phi_c)
                    keep = 1;                   /* first token of its (shifted) window */
            }
            kept[t] = (uint8_t)keep;
            if (keep)
                kv_index[n_kept++] = (int32_t)t;
        }
    }
    frame_off[N] = (int32_t)n_kept;
    return n_kept;
}

/* ---------------------------------------------------------------------------------------
 * Sums of K and V over the dropped set D (one batch element, one head).
 * [AVGGT] Key design 3: one mean key/value stands in for every dropped patch.
 * K, V: [T, d] row-major.  k_sum, v_sum: [d].  Returns the count c = |D|.
 * ------------------------------------------------------------------------------------ */
int64_t oracle_dropped_sums(int64_t T, int d, const uint8_t* kept,
                            const float* K, const float* V, double* k_sum, double* v_sum)
{
    int64_t c = 0;
    for (int j = 0; j < d; ++j) { k_sum[j] = 0.0; v_sum[j] = 0.0; }
    for (int64_t t = 0; t < T; ++t) {
        if (kept[t]) continue;
        ++c;
        for (int j = 0; j < d; ++j) {
            k_sum[j] += (double)K[t * d + j];
            v_sum[j] += (double)V[t * d + j];
        }
    }
    return c;
}

static double dot_fd(const float* a, const float* b, int d)
{
    double s = 0.0;
    for (int j = 0; j < d; ++j) s += (double)a[j] * (double)b[j];
    return s;
}

static double dot_fdd(const float* a, const double* b, int d)
{
    double s = 0.0;
    for (int j = 0; j < d; ++j) s += (double)a[j] * b[j];
    return s;
}

/* ---------------------------------------------------------------------------------------
 * SGA output for selected query rows of one (batch, head).
 * [AVGGT] Key design 2 (attention over S, all queries kept) and Key design 3 (three
 * disjoint components -- S, the diagonal self term, the mean of the dropped set -- under
 * one softmax); [Regime] Key design 2 (the + log(group size) logit bias on a key that
 * stands for several tokens).
 *
 *   Qrows [n_rows, d]  the query vectors of the selected rows
 *   rows  [n_rows]     their token indices in [0, T)
 *   K, V  [T, d]       all keys and values of this head (dropped rows are needed for the
 *                      diagonal term and the leave-one-out mean)
 *   kv_index [S]       the kept set from oracle_plan; kept[T] its indicator
 *   k_sum, v_sum [d], c  from oracle_dropped_sums
 *   diag, mean         switch the two extra components on (1) or off (0)
 *   mean_mode          0 = leave-one-out (reading R5), 1 = global mean over D
 *   out [n_rows, d], lse [n_rows] (nullable)
 * The logits of one row are collected into a buffer, the maximum is subtracted, and the
 * weights are normalised by their sum: a textbook softmax, in fp64.
 * ------------------------------------------------------------------------------------ */
void oracle_sga_rows(int64_t T, int d, const uint8_t* kept, const int32_t* kv_index, int64_t S,
                     const double* k_sum, const double* v_sum, int64_t c,
                     const float* Qrows, const float* K, const float* V,
                     const int64_t* rows, int64_t n_rows,
                     int diag, int mean, int mean_mode, double scale,
                     double* out, double* lse)
{
    #pragma omp parallel
    {
        double* logit = (double*)malloc(sizeof(double) * (size_t)(S + 2));
        double* kbar = (double*)malloc(sizeof(double) * (size_t)d);
        double* vbar = (double*)malloc(sizeof(double) * (size_t)d);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < n_rows; ++n) {
            const int64_t i = rows[n];
            const float* q = Qrows + n * d;
            double* o = out + n * d;

            /* component (i): every kept key */
            for (int64_t s = 0; s < S; ++s)
                logit[s] = scale * dot_fd(q, K + (int64_t)kv_index[s] * d, d);

            /* component (ii): the query's own key, when the query's token was dropped */
            const int has_diag = diag && !kept[i];
            if (has_diag)
                logit[S] = scale * dot_fd(q, K + i * d, d);

            /* component (iii): one mean key/value over the dropped set, logit + ln(count) */
            int64_t ci = c;
            if (mean_mode == 0 && !kept[i]) ci = c - 1;           /* leave i out */
            const int has_mean = mean && ci > 0;
            if (has_mean) {
                for (int j = 0; j < d; ++j) {
                    double ks = k_sum[j], vs = v_sum[j];
                    if (mean_mode == 0 && !kept[i]) {
                        ks -= (double)K[i * d + j];
                        vs -= (double)V[i * d + j];
                    }
                    kbar[j] = ks / (double)ci;
                    vbar[j] = vs / (double)ci;
                }
                logit[S + 1] = scale * dot_fdd(q, kbar, d) + log((double)ci);
            }

            /* one shared softmax over the three components */
            double m = -INFINITY;
            for (int64_t s = 0; s < S; ++s) if (logit[s] > m) m = logit[s];
            if (has_diag && logit[S] > m) m = logit[S];
            if (has_mean && logit[S + 1] > m) m = logit[S + 1];

            double l = 0.0;
            for (int j = 0; j < d; ++j) o[j] = 0.0;
            for (int64_t s = 0; s < S; ++s) {
                const double w = exp(logit[s] - m);
                const float* v = V + (int64_t)kv_index[s] * d;
                l += w;
                for (int j = 0; j < d; ++j) o[j] += w * (double)v[j];
            }
            if (has_diag) {
                const double w = exp(logit[S] - m);
                l += w;
                for (int j = 0; j < d; ++j) o[j] += w * (double)V[i * d + j];
            }
            if (has_mean) {
                const double w = exp(logit[S + 1] - m);
                l += w;
                for (int j = 0; j < d; ++j) o[j] += w * vbar[j];
            }
            for (int j = 0; j < d; ++j) o[j] /= l;
            if (lse) lse[n] = m + log(l);
        }
        free(logit); free(kbar); free(vbar);
    }
}

/* ---------------------------------------------------------------------------------------
 * Textbook attention softmax(q K^T * scale) V for selected rows over the key range
 * [key_lo(i), key_hi(i)).  [AVGGT] Key design 2, the standard attention equation.
 *   frame_len == 0: dense global attention, keys [0, T)
 *   frame_len  > 0: frame-local attention ([AVGGT] Key design 1, Global-to-Frame):
 *                   keys of the query's own frame, [f*frame_len, (f+1)*frame_len)
 * ------------------------------------------------------------------------------------ */
void oracle_attention_rows(int64_t T, int d, int64_t frame_len,
                           const float* Qrows, const float* K, const float* V,
                           const int64_t* rows, int64_t n_rows, double scale,
                           double* out, double* lse)
{
    #pragma omp parallel
    {
        const int64_t cap = frame_len > 0 ? frame_len : T;
        double* logit = (double*)malloc(sizeof(double) * (size_t)cap);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < n_rows; ++n) {
            const int64_t i = rows[n];
            const float* q = Qrows + n * d;
            double* o = out + n * d;
            int64_t lo = 0, hi = T;
            if (frame_len > 0) {
                lo = (i / frame_len) * frame_len;
                hi = lo + frame_len;
            }
            double m = -INFINITY;
            for (int64_t t = lo; t < hi; ++t) {
                logit[t - lo] = scale * dot_fd(q, K + t * d, d);
                if (logit[t - lo] > m) m = logit[t - lo];
            }
            double l = 0.0;
            for (int j = 0; j < d; ++j) o[j] = 0.0;
            for (int64_t t = lo; t < hi; ++t) {
                const double w = exp(logit[t - lo] - m);
                l += w;
                for (int j = 0; j < d; ++j) o[j] += w * (double)V[t * d + j];
            }
            for (int j = 0; j < d; ++j) o[j] /= l;
            if (lse) lse[n] = m + log(l);
        }
        free(logit);
    }
}

/* Threads the OpenMP runtime will use (reported beside CPU timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------------------
 * Size-aware attention, softmax(scale * q K^T + b) V, for selected query rows of one
 * (batch, head).  [Regime] Key design 2: a key that stands for g source tokens carries the
 * logit bias log g (natural log), added after the 1/sqrt(d) scaling; b is that per-key bias
 * (any real value; -INFINITY removes the key).
 *   Qrows [n_rows, d]; K, V [Tk, d]; bias [Tk] (fp64); out [n_rows, d]; lse [n_rows] (nullable)
 * Textbook softmax with max subtraction, in fp64.
 * ------------------------------------------------------------------------------------ */
void oracle_biased_attention_rows(int64_t Tk, int d, const float* Qrows, const float* K,
                                  const float* V, const double* bias, int64_t n_rows,
                                  double scale, double* out, double* lse)
{
    #pragma omp parallel
    {
        double* logit = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t n = 0; n < n_rows; ++n) {
            const float* q = Qrows + n * d;
            double* o = out + n * d;
            double m = -INFINITY;
            for (int64_t t = 0; t < Tk; ++t) {
                logit[t] = scale * dot_fd(q, K + t * d, d) + bias[t];
                if (logit[t] > m) m = logit[t];
            }
            double l = 0.0;
            for (int j = 0; j < d; ++j) o[j] = 0.0;
            for (int64_t t = 0; t < Tk; ++t) {
                const double w = exp(logit[t] - m);
                l += w;
                for (int j = 0; j < d; ++j) o[j] += w * (double)V[t * d + j];
            }
            for (int j = 0; j < d; ++j) o[j] /= l;
            if (lse) lse[n] = m + log(l);
        }
        free(logit);
    }
}

/* ---------------------------------------------------------------------------------------
 * Generalised kept set.  [Regime] Key design 3: per-axis sampling factors that need not be
 * integers (1.5 / 1.3 / 1.7, keeping about 1/sigma_b^2 of the patches), the phase shift,
 * frame 0 and the camera/register tokens at full density, and an externally chosen list of
 * protected (salient) tokens kept in full as well.
 *
 * A window size is the rational sigma = num/den >= 1 (exact integer arithmetic).  Along one
 * axis of length G, window i covers [i*sigma, (i+1)*sigma) and keeps its first position
 * ceil(i*sigma); with the phase shift the positions move by phi, phi + ceil(i*sigma) < G.
 * The phase uses the page's formula with the integer tile t = ceil(sigma) per axis:
 * phi_r = (f div t_w) mod t_h, phi_c = f mod t_w (for integer sigma this is the plain grid).
 * protected_tokens: n_protected token indices in [0, N*L), any order, repeats allowed.
 * Outputs as oracle_plan.  Returns |S|, or -1 on a bad argument.
 * ------------------------------------------------------------------------------------ */
static int on_axis(int64_t x, int64_t phi, int64_t num, int64_t den)
{
    /* is x = phi + ceil(i * num / den) for some integer i >= 0 ? */
    if (x < phi) return 0;
    const int64_t y = x - phi;
    if (y == 0) return 1;
    /* ceil(i*sigma) >= y  <=>  i*sigma > y - 1: the smallest such i is floor((y-1)/sigma) + 1;
       y is a window start iff that window starts exactly at y */
    const int64_t i = ((y - 1) * den) / num + 1;
    return (i * num + den - 1) / den == y;
}

int64_t oracle_plan_general(int N, int grid_h, int grid_w, int n_special,
                            int sh_num, int sh_den, int sw_num, int sw_den,
                            int phase_shift, int ref_frame_dense,
                            const int32_t* protected_tokens, int64_t n_protected,
                            uint8_t* kept, int32_t* kv_index, int32_t* frame_off)
{
    if (N <= 0 || grid_h <= 0 || grid_w <= 0 || n_special < 0 || sh_den <= 0 || sw_den <= 0 ||
        sh_num < sh_den || sw_num < sw_den || n_protected < 0)
        return -1;
    const int64_t L = (int64_t)n_special + (int64_t)grid_h * grid_w;
    const int64_t T = (int64_t)N * L;
    const int64_t th = (sh_num + sh_den - 1) / sh_den, tw = (sw_num + sw_den - 1) / sw_den;
    for (int64_t t = 0; t < T; ++t) kept[t] = 0;
    for (int64_t k = 0; k < n_protected; ++k) {
        if (protected_tokens[k] < 0 || protected_tokens[k] >= T) return -1;
        kept[protected_tokens[k]] = 1;                 /* protected salient token */
    }
    int64_t n_kept = 0;
    for (int f = 0; f < N; ++f) {
        frame_off[f] = (int32_t)n_kept;
        int64_t phi_r = 0, phi_c = 0;
        if (phase_shift) {
            phi_r = (f / tw) % th;
            phi_c = f % tw;
        }
        for (int64_t p = 0; p < L; ++p) {
            const int64_t t = (int64_t)f * L + p;
            if (f == 0 && ref_frame_dense) {
                kept[t] = 1;                           /* reference frame uncompressed */
            } else if (p < n_special) {
                kept[t] = 1;                           /* camera / register tokens */
            } else {
                const int64_t r = (p - n_special) / grid_w;
                const int64_t c = (p - n_special) % grid_w;
                if (on_axis(r, phi_r, sh_num, sh_den) && on_axis(c, phi_c, sw_num, sw_den))
                    kept[t] = 1;                       /* first position of its window */
            }
            if (kept[t])
                kv_index[n_kept++] = (int32_t)t;
        }
    }
    frame_off[N] = (int32_t)n_kept;
    return n_kept;
}

/* ---------------------------------------------------------------------------------------
 * 2D rotary position embedding of one (batch, head)'s tokens, the step before the attention:
 * VGGT re-applies rotary position encoding to Q and K in every layer ("HTTM: Head-wise Temporal
 * Token Merging for Faster VGGT", blog digest, section 3 "core insight: VGGT's token similarity
 * patterns", the RoPE architecture effect).  The pages give no frequency convention, so it is
 * parametrised here (the same reading in the CUDA path):
 *   dims [0, d/2) rotate by the row position, dims [d/2, d) by the column position;
 *   within a half of size h = d/2 the pairs (j, j + h/2), j < h/2, rotate by the angle
 *   pos * base^(-2j/h);
 *   a patch (r, c) sits at (r + pos_offset, c + pos_offset); the n_special camera/register
 *   tokens sit at position 0 (no rotation).
 * X: [T, d] in (fp32), Y: [T, d] out (fp64); T = N * L, L = n_special + grid_h * grid_w.
 * ------------------------------------------------------------------------------------ */
void oracle_rope2d(int64_t T, int d, int64_t L, int n_special, int grid_w, double base,
                   int pos_offset, const float* X, double* Y)
{
    const int h = d / 2, q = h / 2;
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const int64_t p = t % L;
        double pos[2] = {0.0, 0.0};
        if (p >= n_special) {
            pos[0] = (double)((p - n_special) / grid_w + pos_offset);   /* row */
            pos[1] = (double)((p - n_special) % grid_w + pos_offset);   /* column */
        }
        for (int a = 0; a < 2; ++a) {
            for (int j = 0; j < q; ++j) {
                const double ang = pos[a] * pow(base, -2.0 * j / h);
                const double x0 = (double)X[t * d + a * h + j];
                const double x1 = (double)X[t * d + a * h + j + q];
                Y[t * d + a * h + j] = x0 * cos(ang) - x1 * sin(ang);
                Y[t * d + a * h + j + q] = x0 * sin(ang) + x1 * cos(ang);
            }
        }
    }
}

/* ---------------------------------------------------------------------------------------
 * Head-wise temporal token merging ("HTTM: Head-wise Temporal Token Merging for Faster VGGT",
 * blog digest, section 2 "core method": head-wise merging, temporal reordering and block-level
 * merging, first-frame anchoring; "RegimeVGGT ..." Key design 1-2: merged keys carry log g).
 * One (batch, head), tokens X [T, d] (the keys; the values follow the keys' matching).
 *
 * Reading (where the pages leave the details open):
 *   - frames are grouped in chunks of n_t consecutive frames; a block is the same run of n_s
 *     consecutive patch tokens (row-major, the last run of a frame may be shorter) in every
 *     frame of one chunk;
 *   - in a block, the tokens of the chunk's first frame are the destinations (anchors), the
 *     tokens of its other frames the sources; special tokens are never merged;
 *   - each source s is matched to the destination d with the largest cosine similarity (ties:
 *     the lowest token index); the r = floor(|sources| * r_permille / 1000) sources with the
 *     largest similarity (ties: lowest token index) are merged into their destination;
 *   - the cosine is decided in IEEE fp32 with one fixed operation order (the same in the CUDA
 *     kernel): n_x = sqrt(fma-chain of x_i^2, i = 0..d-1), dot = fma-chain of x_i y_i,
 *     cos = dot / (n_s * n_d), and 0 when n_s * n_d == 0.
 * Output: match[t] = destination token of a merged source t, else -1.  Returns the number of
 * merged sources, or -1 on a bad argument.
 * ------------------------------------------------------------------------------------ */
static float cos_f32(const float* x, const float* y, int d, float nx, float ny)
{
    float dot = 0.0f;
    for (int i = 0; i < d; ++i) dot = fmaf(x[i], y[i], dot);
    const float den = nx * ny;
    return den == 0.0f ? 0.0f : dot / den;
}

static float norm_f32(const float* x, int d)
{
    float s = 0.0f;
    for (int i = 0; i < d; ++i) s = fmaf(x[i], x[i], s);
    return sqrtf(s);
}

int64_t oracle_merge_match(int N, int grid_h, int grid_w, int n_special, int n_t, int n_s,
                           int r_permille, int d, const float* X, int32_t* match)
{
    if (N <= 0 || grid_h <= 0 || grid_w <= 0 || n_special < 0 || n_t <= 0 || n_s <= 0 ||
        r_permille < 0 || r_permille > 1000)
        return -1;
    const int64_t P = (int64_t)grid_h * grid_w, L = n_special + P, T = (int64_t)N * L;
    for (int64_t t = 0; t < T; ++t) match[t] = -1;
    int64_t merged = 0;
    float* sim = (float*)malloc(sizeof(float) * (size_t)(n_t * n_s));
    int64_t* best = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_t * n_s));
    int64_t* src = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_t * n_s));
    for (int f0 = 0; f0 < N; f0 += n_t) {
        const int nf = (f0 + n_t <= N) ? n_t : N - f0;
        for (int64_t w0 = 0; w0 < P; w0 += n_s) {
            const int64_t ws = (w0 + n_s <= P) ? n_s : P - w0;
            /* match every source of the block (frames f0+1 .. f0+nf-1) to a destination */
            int64_t n_src = 0;
            for (int f = f0 + 1; f < f0 + nf; ++f) {
                for (int64_t k = 0; k < ws; ++k) {
                    const int64_t s = (int64_t)f * L + n_special + w0 + k;
                    const float ns = norm_f32(X + s * d, d);
                    float bs = -INFINITY;
                    int64_t bd = -1;
                    for (int64_t k2 = 0; k2 < ws; ++k2) {
                        const int64_t dd = (int64_t)f0 * L + n_special + w0 + k2;
                        const float c = cos_f32(X + s * d, X + dd * d, d, ns, norm_f32(X + dd * d, d));
                        if (c > bs) { bs = c; bd = dd; }       /* strict: the first maximum wins */
                    }
                    src[n_src] = s;
                    sim[n_src] = bs;
                    best[n_src] = bd;
                    ++n_src;
                }
            }
            /* merge the r most similar sources: rank = number of sources ahead of s */
            const int64_t r = n_src * r_permille / 1000;
            for (int64_t a = 0; a < n_src; ++a) {
                int64_t rank = 0;
                for (int64_t b = 0; b < n_src; ++b)
                    if (sim[b] > sim[a] || (sim[b] == sim[a] && src[b] < src[a])) ++rank;
                if (rank < r) {
                    match[src[a]] = (int32_t)best[a];
                    ++merged;
                }
            }
        }
    }
    free(sim); free(best); free(src);
    return merged;
}
