/*
 * CPU oracle for the time-unrolled recurrent-cell forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Everything here is plain fp64 arithmetic over the recurrence as written,
 * one batch row at a time (rows are independent), with no blocking, fusion
 * or reordering.  Inputs arrive as the same fp32 bits the GPU receives and
 * are widened to double; for the bf16-weight path the weights are first
 * rounded to bf16 (round-to-nearest-even) so that weight quantisation is not
 * counted as error.
 *
 * Sources for what is computed (the pages name the modules, not their
 * equations; the equations are the standard ones of the modules named):
 *  - LSTM / LSTM with projection: "Integrating CuDNN API for LSTMs with
 *    projections" (pytorch/pytorch issue 46213), Pitch and the design reply
 *    on CellParams: the projected cell is the ordinary LSTM cell followed by
 *    one more matmul on the resulting hidden state (h = W_hr (o * tanh c)).
 *  - GRU: the nn.GRUCell named as the core of RSSMPrior in
 *    "[Feature Request] CUDNN version of RSSM" (pytorch/rl issue 366),
 *    Motivation and Solution; reset gate applied after the hidden matmul.
 *  - Variable-length batches, sort by length and packing: "RNN Op Changes
 *    (was: Variable Length Support for cuDNN RNN)" (apache/mxnet issue 9543),
 *    first post.  Ties in the length sort keep ascending row order.
 *  - RSSM prior step and unroll variant 1: pytorch/rl issue 366, Solution
 *    (RSSMPrior.forward and the first unroll_rssm), with the noise supplied
 *    as an input tensor and the NormalParamWrapper read as
 *    mean = p[:S], std = softplus(p[S:]) + scale_lb (scale_lb = 0.1).
 *
 * Pins: every function here is checked in tests/test_oracle_pins.py against
 * closed forms, saturated-gate limits, hand-computed single steps, an
 * independently written scalar Python evaluation on tiny inputs, invariants
 * (batch permutation, composition of layers, packed == per-sequence), and an
 * independent library evaluation (torch float64 on CPU).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_LSTM 0
#define OR_GRU 1

/* Weights of one layer and direction, PyTorch layout, fp32 bits. */
typedef struct {
    const float *w_ih; /* [nG*H, in]   */
    const float *w_hh; /* [nG*H, Hout] */
    const float *b_ih; /* [nG*H] or NULL (= zero) */
    const float *b_hh; /* [nG*H] or NULL (= zero) */
    const float *w_hr; /* [P, H] or NULL when there is no projection */
} oracle_layer_w;

/* fp32 -> bf16 -> fp32 with round-to-nearest-even on the bit pattern. */
static double bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {          /* inf or nan */
        if (u & 0x007fffffu) u |= 0x00400000u;        /* quiet nan */
        u &= 0xffff0000u;
    } else {
        uint32_t keep_lsb = (u >> 16) & 1u;
        u += 0x7fffu + keep_lsb;
        u &= 0xffff0000u;
    }
    float r;
    memcpy(&r, &u, sizeof r);
    return (double)r;
}

/* Widen n fp32 values to double, optionally through bf16 first. NULL -> zeros. */
static double *widen(const float *src, size_t n, int to_bf16) {
    double *d = (double *)calloc(n ? n : 1, sizeof(double));
    if (!d) return NULL;
    if (src)
        for (size_t i = 0; i < n; ++i) d[i] = to_bf16 ? bf16_rne(src[i]) : (double)src[i];
    return d;
}

double oracle_bf16_round(float f) { return bf16_rne(f); }

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }
static double elu(double v) { return v > 0.0 ? v : expm1(v); }
static double softplus(double v) { return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v))); }

/* ---------------------------------------------------------------------- */
/* Length sort and packing metadata.                                        */
/* sorted_idx[s]  = original row at sorted position s, ordered by length   */
/*                  descending, ties by ascending original index;          */
/* unsorted_idx[b] = sorted position of original row b;                    */
/* batch_sizes[t] = number of rows whose length exceeds t.                 */
/* Returns -1 if some length is outside [1, T].                             */
int oracle_pack(int B, int T, const int32_t *lengths, int32_t *sorted_idx,
                int32_t *unsorted_idx, int32_t *batch_sizes) {
    for (int b = 0; b < B; ++b)
        if (lengths[b] < 1 || lengths[b] > T) return -1;
    /* plain selection: position of row b = rows that must come before it */
    for (int b = 0; b < B; ++b) {
        int pos = 0;
        for (int o = 0; o < B; ++o)
            if (lengths[o] > lengths[b] || (lengths[o] == lengths[b] && o < b)) ++pos;
        sorted_idx[pos] = b;
        unsorted_idx[b] = pos;
    }
    for (int t = 0; t < T; ++t) {
        int n = 0;
        for (int b = 0; b < B; ++b)
            if (lengths[b] > t) ++n;
        batch_sizes[t] = n;
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* One direction of one layer for one batch row.                            */
/* in_seq: [len][in_w] input vectors of this row (time order);             */
/* out:    [T][out_stride] written at column offset col for t < len.       */
/* h, c:   state, updated in place (c unused for GRU).                     */
/* clip: NULL, or {cell_lo, cell_hi, proj_lo, proj_hi}: the LSTM cell state
   is clamped to [cell_lo, cell_hi] as soon as it is updated (before tanh),
   the projected hidden state to [proj_lo, proj_hi] as soon as it is formed
   (cell-state and projection clipping of cuDNN 7.2, "RNN Op Changes",
   apache/mxnet issue 9543). */
static double clampd(double v, double lo, double hi) { return v < lo ? lo : (v > hi ? hi : v); }

static void run_direction(int cell, int in_w, int H, int P, int len, int reverse,
                          const double *in_seq, const double *Wih, const double *Whh,
                          const double *bih, const double *bhh, const double *Whr,
                          double *h, double *c, double *out, int out_stride, int col,
                          double *scratch /* [nG*H + H] */, const double *clip) {
    const int nG = (cell == OR_LSTM) ? 4 : 3;
    const int Hout = P > 0 ? P : H;
    double *pre = scratch;          /* nG*H */
    double *m = scratch + nG * H;   /* H */
    for (int s = 0; s < len; ++s) {
        const int t = reverse ? (len - 1 - s) : s;
        const double *xt = in_seq + (size_t)t * in_w;
        if (cell == OR_LSTM) {
            /* gates = W_ih x + b_ih + W_hh h + b_hh, rows ordered i, f, g, o */
            for (int r = 0; r < nG * H; ++r) {
                double acc = bih[r] + bhh[r];
                for (int k = 0; k < in_w; ++k) acc += Wih[(size_t)r * in_w + k] * xt[k];
                for (int k = 0; k < Hout; ++k) acc += Whh[(size_t)r * Hout + k] * h[k];
                pre[r] = acc;
            }
            for (int j = 0; j < H; ++j) {
                double ig = sigmoid(pre[0 * H + j]);
                double fg = sigmoid(pre[1 * H + j]);
                double gg = tanh(pre[2 * H + j]);
                double og = sigmoid(pre[3 * H + j]);
                c[j] = fg * c[j] + ig * gg;
                if (clip) c[j] = clampd(c[j], clip[0], clip[1]);
                m[j] = og * tanh(c[j]);
            }
            if (P > 0) {
                /* projected hidden state h = W_hr m (no bias) */
                for (int p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int j = 0; j < H; ++j) acc += Whr[(size_t)p * H + j] * m[j];
                    h[p] = clip ? clampd(acc, clip[2], clip[3]) : acc;
                }
            } else {
                for (int j = 0; j < H; ++j) h[j] = m[j];
            }
        } else {
            /* GRU, rows ordered r, z, n; the reset gate multiplies the
               hidden-side n pre-activation including its bias */
            double *gi = pre; /* staging for the new h, H entries */
            for (int j = 0; j < H; ++j) {
                double ir = bih[0 * H + j], iz = bih[1 * H + j], in_ = bih[2 * H + j];
                double hr = bhh[0 * H + j], hz = bhh[1 * H + j], hn = bhh[2 * H + j];
                for (int k = 0; k < in_w; ++k) {
                    ir += Wih[(size_t)(0 * H + j) * in_w + k] * xt[k];
                    iz += Wih[(size_t)(1 * H + j) * in_w + k] * xt[k];
                    in_ += Wih[(size_t)(2 * H + j) * in_w + k] * xt[k];
                }
                for (int k = 0; k < H; ++k) {
                    hr += Whh[(size_t)(0 * H + j) * H + k] * h[k];
                    hz += Whh[(size_t)(1 * H + j) * H + k] * h[k];
                    hn += Whh[(size_t)(2 * H + j) * H + k] * h[k];
                }
                double rg = sigmoid(ir + hr);
                double zg = sigmoid(iz + hz);
                double ng = tanh(in_ + rg * hn);
                gi[j] = (1.0 - zg) * ng + zg * h[j]; /* new h, staged */
            }
            for (int j = 0; j < H; ++j) h[j] = gi[j];
        }
        double *ot = out + (size_t)t * out_stride + col;
        for (int k = 0; k < Hout; ++k) ot[k] = h[k];
    }
}

/*
 * Full forward of a stacked (optionally bidirectional, optionally projected)
 * LSTM or GRU, restricted to the batch rows listed in `rows` (all rows when
 * rows == NULL).  Rows are independent, so the restriction computes exactly
 * the same values for the listed rows.
 *
 * x        [T, B, in]          fp32
 * lengths  [B] or NULL (all T)
 * h0       [L*D, B, Hout] or NULL (zeros);  c0 [L*D, B, H] or NULL (zeros)
 * w        [L*D] weight sets, index l*D + d
 * y        [T, B, D*Hout] double; rows listed are fully written (zeros past length)
 * h_n      [L*D, B, Hout] double or NULL;  c_n [L*D, B, H] double or NULL
 * Returns 0, or -1 on invalid arguments.
 */
int oracle_rnn_forward(int cell, int bidir, int layers, int in_dim, int hidden, int proj,
                       int bf16_weights, int T, int B, const float *x, const int32_t *lengths,
                       const float *h0, const float *c0, const oracle_layer_w *w, double *y,
                       double *h_n, double *c_n, const int32_t *rows, int nrows, int nthreads,
                       const double *clip) {
    if (cell != OR_LSTM && cell != OR_GRU) return -1;
    if (layers < 1 || in_dim < 1 || hidden < 1 || T < 0 || B < 0) return -1;
    if (proj < 0 || (proj > 0 && cell != OR_LSTM)) return -1;
    const int D = bidir ? 2 : 1;
    const int H = hidden, P = proj, Hout = proj > 0 ? proj : hidden;
    const int nG = (cell == OR_LSTM) ? 4 : 3;
    if (lengths)
        for (int b = 0; b < B; ++b)
            if (lengths[b] < 1 || lengths[b] > T) return -1;
    const int nsel = rows ? nrows : B;

    /* widen all weights once (shared read-only by all threads) */
    const int LD = layers * D;
    double **Wih = (double **)calloc(LD, sizeof(double *));
    double **Whh = (double **)calloc(LD, sizeof(double *));
    double **bih = (double **)calloc(LD, sizeof(double *));
    double **bhh = (double **)calloc(LD, sizeof(double *));
    double **Whr = (double **)calloc(LD, sizeof(double *));
    for (int l = 0; l < layers; ++l) {
        const int in_w = (l == 0) ? in_dim : D * Hout;
        for (int d = 0; d < D; ++d) {
            const int i = l * D + d;
            Wih[i] = widen(w[i].w_ih, (size_t)nG * H * in_w, bf16_weights);
            Whh[i] = widen(w[i].w_hh, (size_t)nG * H * Hout, bf16_weights);
            /* biases stay fp32 on both paths */
            bih[i] = widen(w[i].b_ih, (size_t)nG * H, 0);
            bhh[i] = widen(w[i].b_hh, (size_t)nG * H, 0);
            Whr[i] = P > 0 ? widen(w[i].w_hr, (size_t)P * H, bf16_weights) : NULL;
        }
    }

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        const int wmax = (in_dim > D * Hout ? in_dim : D * Hout);
        double *seq_a = (double *)malloc((size_t)(T ? T : 1) * wmax * sizeof(double));
        double *seq_b = (double *)malloc((size_t)(T ? T : 1) * D * Hout * sizeof(double));
        double *h = (double *)malloc((size_t)Hout * sizeof(double));
        double *c = (double *)malloc((size_t)H * sizeof(double));
        double *scratch = (double *)malloc((size_t)(nG * H + H + nG * H) * sizeof(double));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int q = 0; q < nsel; ++q) {
            const int b = rows ? rows[q] : q;
            const int len = lengths ? lengths[b] : T;
            /* layer-0 input sequence of this row */
            for (int t = 0; t < len; ++t)
                for (int k = 0; k < in_dim; ++k)
                    seq_a[(size_t)t * in_dim + k] = (double)x[((size_t)t * B + b) * in_dim + k];
            int in_w = in_dim;
            for (int l = 0; l < layers; ++l) {
                for (int d = 0; d < D; ++d) {
                    const int i = l * D + d;
                    for (int k = 0; k < Hout; ++k)
                        h[k] = h0 ? (double)h0[((size_t)i * B + b) * Hout + k] : 0.0;
                    for (int k = 0; k < H; ++k)
                        c[k] = c0 ? (double)c0[((size_t)i * B + b) * H + k] : 0.0;
                    run_direction(cell, in_w, H, P, len, d == 1, seq_a, Wih[i], Whh[i], bih[i],
                                  bhh[i], Whr[i], h, c, seq_b, D * Hout, d * Hout, scratch, clip);
                    if (h_n)
                        for (int k = 0; k < Hout; ++k) h_n[((size_t)i * B + b) * Hout + k] = h[k];
                    if (c_n && cell == OR_LSTM)
                        for (int k = 0; k < H; ++k) c_n[((size_t)i * B + b) * H + k] = c[k];
                }
                /* this layer's output is the next layer's input */
                in_w = D * Hout;
                memcpy(seq_a, seq_b, (size_t)len * in_w * sizeof(double));
            }
            for (int t = 0; t < T; ++t)
                for (int k = 0; k < D * Hout; ++k)
                    y[((size_t)t * B + b) * D * Hout + k] =
                        t < len ? seq_a[(size_t)t * D * Hout + k] : 0.0;
        }
        free(seq_a);
        free(seq_b);
        free(h);
        free(c);
        free(scratch);
    }
    for (int i = 0; i < LD; ++i) {
        free(Wih[i]);
        free(Whh[i]);
        free(bih[i]);
        free(bhh[i]);
        free(Whr[i]);
    }
    free(Wih);
    free(Whh);
    free(bih);
    free(bhh);
    free(Whr);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* RSSM prior unroll with given actions (unroll variant 1).                 */
/*                                                                          */
/* Per step:  a      = ELU(W1 [state, action] + b1)           (width Hd)    */
/*            belief = GRUCell(a, belief)                     (width RH)    */
/*            q      = ELU(W2 belief + b2)                    (width Hd)    */
/*            p      = W3 q + b3                              (width 2S)    */
/*            mean = p[:S];  std = softplus(p[S:]) + 0.1;                   */
/*            state = mean + eps_t * std                                    */
/* Outputs at step t are those after the step's update.                    */
/* Layouts: W1 [Hd, S+A] (state columns first), Wih [3RH, Hd],              */
/* Whh [3RH, RH], W2 [Hd, RH], W3 [2S, Hd]; actions [T,B,A], eps [T,B,S],   */
/* state0 [B,S], belief0 [B,RH] (NULL = zeros); means/stds/states [T,B,S],  */
/* beliefs [T,B,RH].                                                        */
/*                                                                          */
/* Unroll variant 2 ("Given an actor model, we unroll the states for H      */
/* steps computing the actions on the fly", same page): the action of step  */
/* t is actor(state, belief) of the state and belief before the step.  The  */
/* page does not define the actor; it is read here as the plainest model    */
/* in the style of the prior's own projectors, a deterministic two-layer    */
/* MLP:  action = tanh(Wa2 ELU(Wa1 [state, belief] + ba1) + ba2),           */
/* Wa1 [Ha, S+RH] (state columns first), ba1 [Ha], Wa2 [A, Ha], ba2 [A].    */
/* actions_out [T,B,A] receives the actions used (may be NULL).            */
/* With Wa1 == NULL, the actions are read from `actions` (variant 1).       */
int oracle_rssm_unroll2(int S, int A, int Hd, int RH, int T, int B, const float *W1,
                        const float *b1, const float *Wih, const float *Whh, const float *bih,
                        const float *bhh, const float *W2, const float *b2, const float *W3,
                        const float *b3, const float *state0, const float *belief0,
                        const float *actions, const float *eps, double *means, double *stds,
                        double *states, double *beliefs, const int32_t *rows, int nrows,
                        int nthreads, int Ha, const float *Wa1, const float *ba1,
                        const float *Wa2, const float *ba2, double *actions_out) {
    if (S < 1 || A < 0 || Hd < 1 || RH < 1 || T < 0 || B < 0) return -1;
    const int actor = Wa1 != NULL;
    if (actor && (Ha < 1 || !Wa2 || A < 1)) return -1;
    if (!actor && A > 0 && !actions) return -1;
    double *wa1 = actor ? widen(Wa1, (size_t)Ha * (S + RH), 0) : NULL;
    double *vba1 = actor ? widen(ba1, Ha, 0) : NULL;
    double *wa2 = actor ? widen(Wa2, (size_t)A * Ha, 0) : NULL;
    double *vba2 = actor ? widen(ba2, A, 0) : NULL;
    const int nsel = rows ? nrows : B;
    double *w1 = widen(W1, (size_t)Hd * (S + A), 0), *vb1 = widen(b1, Hd, 0);
    double *wih = widen(Wih, (size_t)3 * RH * Hd, 0), *whh = widen(Whh, (size_t)3 * RH * RH, 0);
    double *vbih = widen(bih, (size_t)3 * RH, 0), *vbhh = widen(bhh, (size_t)3 * RH, 0);
    double *w2 = widen(W2, (size_t)Hd * RH, 0), *vb2 = widen(b2, Hd, 0);
    double *w3 = widen(W3, (size_t)2 * S * Hd, 0), *vb3 = widen(b3, (size_t)2 * S, 0);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double *state = (double *)malloc((size_t)S * sizeof(double));
        double *bel = (double *)malloc((size_t)RH * sizeof(double));
        double *nbel = (double *)malloc((size_t)RH * sizeof(double));
        double *a = (double *)malloc((size_t)Hd * sizeof(double));
        double *q = (double *)malloc((size_t)Hd * sizeof(double));
        double *p = (double *)malloc((size_t)2 * S * sizeof(double));
        double *act = (double *)malloc((size_t)(A > 0 ? A : 1) * sizeof(double));
        double *ha = (double *)malloc((size_t)(Ha > 0 ? Ha : 1) * sizeof(double));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int qi = 0; qi < nsel; ++qi) {
            const int b = rows ? rows[qi] : qi;
            for (int j = 0; j < S; ++j) state[j] = state0 ? (double)state0[(size_t)b * S + j] : 0.0;
            for (int j = 0; j < RH; ++j)
                bel[j] = belief0 ? (double)belief0[(size_t)b * RH + j] : 0.0;
            for (int t = 0; t < T; ++t) {
                if (actor) {
                    /* action = actor(state, belief), both before the step */
                    for (int i = 0; i < Ha; ++i) {
                        double u = vba1 ? vba1[i] : 0.0;
                        for (int j = 0; j < S; ++j) u += wa1[(size_t)i * (S + RH) + j] * state[j];
                        for (int j = 0; j < RH; ++j)
                            u += wa1[(size_t)i * (S + RH) + S + j] * bel[j];
                        ha[i] = elu(u);
                    }
                    for (int j = 0; j < A; ++j) {
                        double v = vba2 ? vba2[j] : 0.0;
                        for (int i = 0; i < Ha; ++i) v += wa2[(size_t)j * Ha + i] * ha[i];
                        act[j] = tanh(v);
                    }
                } else {
                    for (int j = 0; j < A; ++j) act[j] = (double)actions[((size_t)t * B + b) * A + j];
                }
                if (actions_out)
                    for (int j = 0; j < A; ++j) actions_out[((size_t)t * B + b) * A + j] = act[j];
                for (int i = 0; i < Hd; ++i) {
                    double u = vb1[i];
                    for (int j = 0; j < S; ++j) u += w1[(size_t)i * (S + A) + j] * state[j];
                    for (int j = 0; j < A; ++j) u += w1[(size_t)i * (S + A) + S + j] * act[j];
                    a[i] = elu(u);
                }
                for (int j = 0; j < RH; ++j) {
                    double ir = vbih[j], iz = vbih[RH + j], in_ = vbih[2 * RH + j];
                    double hr = vbhh[j], hz = vbhh[RH + j], hn = vbhh[2 * RH + j];
                    for (int k = 0; k < Hd; ++k) {
                        ir += wih[(size_t)j * Hd + k] * a[k];
                        iz += wih[(size_t)(RH + j) * Hd + k] * a[k];
                        in_ += wih[(size_t)(2 * RH + j) * Hd + k] * a[k];
                    }
                    for (int k = 0; k < RH; ++k) {
                        hr += whh[(size_t)j * RH + k] * bel[k];
                        hz += whh[(size_t)(RH + j) * RH + k] * bel[k];
                        hn += whh[(size_t)(2 * RH + j) * RH + k] * bel[k];
                    }
                    double rg = sigmoid(ir + hr), zg = sigmoid(iz + hz);
                    double ng = tanh(in_ + rg * hn);
                    nbel[j] = (1.0 - zg) * ng + zg * bel[j];
                }
                memcpy(bel, nbel, (size_t)RH * sizeof(double));
                for (int i = 0; i < Hd; ++i) {
                    double v = vb2[i];
                    for (int k = 0; k < RH; ++k) v += w2[(size_t)i * RH + k] * bel[k];
                    q[i] = elu(v);
                }
                for (int i = 0; i < 2 * S; ++i) {
                    double v = vb3[i];
                    for (int k = 0; k < Hd; ++k) v += w3[(size_t)i * Hd + k] * q[k];
                    p[i] = v;
                }
                const size_t o = ((size_t)t * B + b) * S;
                for (int j = 0; j < S; ++j) {
                    const double mean = p[j];
                    const double sd = softplus(p[S + j]) + 0.1;
                    state[j] = mean + (double)eps[o + j] * sd;
                    means[o + j] = mean;
                    stds[o + j] = sd;
                    states[o + j] = state[j];
                }
                for (int j = 0; j < RH; ++j) beliefs[((size_t)t * B + b) * RH + j] = bel[j];
            }
        }
        free(state);
        free(bel);
        free(nbel);
        free(a);
        free(q);
        free(p);
        free(act);
        free(ha);
    }
    free(w1); free(vb1); free(wih); free(whh); free(vbih); free(vbhh);
    free(w2); free(vb2); free(w3); free(vb3);
    free(wa1); free(vba1); free(wa2); free(vba2);
    return 0;
}

/* Unroll variant 1 (actions given). */
int oracle_rssm_unroll(int S, int A, int Hd, int RH, int T, int B, const float *W1,
                       const float *b1, const float *Wih, const float *Whh, const float *bih,
                       const float *bhh, const float *W2, const float *b2, const float *W3,
                       const float *b3, const float *state0, const float *belief0,
                       const float *actions, const float *eps, double *means, double *stds,
                       double *states, double *beliefs, const int32_t *rows, int nrows,
                       int nthreads) {
    return oracle_rssm_unroll2(S, A, Hd, RH, T, B, W1, b1, Wih, Whh, bih, bhh, W2, b2, W3, b3,
                               state0, belief0, actions, eps, means, stds, states, beliefs, rows,
                               nrows, nthreads, 0, NULL, NULL, NULL, NULL, NULL);
}

int oracle_num_threads_default(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------- */
/* Backward pass through time (BPTT) of the stacked unidirectional          */
/* LSTM / GRU, optionally LSTM with projection: the training use of the    */
/* unrolled cell behind the RSSM page's                                     */
/* Motivation and the LSTMP page's training discussion.  The gradient of a  */
/* scalar loss whose derivative with respect to y is dy [T,B,Ho] (and to    */
/* h_n / c_n is dh_n [L,B,Ho] / dc_n [L,B,H], NULL = 0; Ho = proj or H) is  */
/* taken through the forward recurrence exactly as written above, in       */
/* reverse time, by the chain rule:                                         */
/*   LSTM  m = o tanh(c),  c = f c' + i g,  h = W_hr m (projection) or m:    */
/*     dm = W_hr^T dh (projection; dW_hr += dh m^T) or dh;                  */
/*     do = dm tanh(c);  dc += dm o (1 - tanh^2 c);                         */
/*     di = dc g;  df = dc c';  dg = dc i;  dc' = dc f;                     */
/*     dz = [di i(1-i), df f(1-f), dg (1-g^2), do o(1-o)]  (pre-activations)*/
/*     dx_t = W_ih^T dz;  dh' = W_hh^T dz;  dW_ih += dz x^T;               */
/*     dW_hh += dz h'^T;  db_ih += dz;  db_hh += dz                          */
/*   GRU  h = (1-z) n + z h',  n = tanh(a_n + r hn),  hn = W_hn h' + b_hn:   */
/*     dn = dh (1-z);  dz = dh (h' - n);  dh' = dh z (direct);              */
/*     dan = dn (1-n^2);  dr = dan hn;  dhn = dan r;                        */
/*     input side  dA = [dr r(1-r), dz z(1-z), dan]                         */
/*     hidden side dR = [dr r(1-r), dz z(1-z), dhn]                         */
/*     dx_t = W_ih^T dA;  dh' += W_hh^T dR;  dW_ih += dA x^T;              */
/*     dW_hh += dR h'^T;  db_ih += dA;  db_hh += dR                          */
/* Bidirectional: direction 1 runs its forward from t = T-1 down to 0, so   */
/* its backward replays t = 0 .. T-1; layer l+1's input is [h_fwd, h_bwd]  */
/* and both directions' input gradients add into layer l's dy.             */
/* Layer l's dx is layer l-1's dy.  Weight gradients are summed over rows   */
/* and steps; layouts follow the weights per (layer, direction) i = l*D + d */
/* (dW_ih at offset sum_{j<i} nG*H*in_j, dW_hh at i*nG*H*Ho, db at i*nG*H,  */
/* dW_hr at i*P*H).  Outputs: dx [T,B,in], dh0 [L*D,B,Ho], dc0 [L*D,B,H]    */
/* (LSTM; may be NULL).  lengths: NULL or [B] in [1, T]: row b runs steps    */
/* t < len_b as in the forward (the backward direction from len_b - 1), its */
/* dh_n enters at its last processed step and dx is 0 at t >= len_b.        */
/* bf16_weights: the weight matrices are first rounded                     */
/* to bf16 (the forward oracle's convention; biases stay fp32).             */
/* clip: NULL or {cell_lo, cell_hi, proj_lo, proj_hi} as in the forward     */
/* (LSTM only): a clamp passes the gradient where the unclamped value lies  */
/* in [lo, hi] (bounds included) and stops it elsewhere, so dc and dh are   */
/* masked by that condition right after they reach the clamped value.       */
int oracle_rnn_backward(int cell, int bidir, int layers, int in_dim, int hidden, int proj,
                        int bf16_weights, int T, int B, const float *x, const int32_t *lengths,
                        const float *h0, const float *c0,
                        const oracle_layer_w *w, const float *dy, const float *dh_n,
                        const float *dc_n, double *dx, double *dh0, double *dc0, double *dW_ih,
                        double *dW_hh, double *db_ih, double *db_hh, double *dW_hr,
                        int nthreads, const double *clip) {
    if (cell != OR_LSTM && cell != OR_GRU) return -1;
    if (clip && cell != OR_LSTM) return -1;
    if (layers < 1 || in_dim < 1 || hidden < 1 || T < 1 || B < 1 || !x || !dy) return -1;
    if (proj < 0 || (proj > 0 && cell != OR_LSTM)) return -1;
    if (lengths)
        for (int b = 0; b < B; ++b)
            if (lengths[b] < 1 || lengths[b] > T) return -1;
    const int D = bidir ? 2 : 1, LD = layers * D;
    const int H = hidden, P = proj, Ho = proj > 0 ? proj : hidden, DHo = D * Ho;
    const int nG = (cell == OR_LSTM) ? 4 : 3, G = nG * H;
    const int lstm = cell == OR_LSTM;
    /* per (layer, direction) i = l*D + d */
    size_t *off_ih = (size_t *)calloc((size_t)LD + 1, sizeof(size_t));
    double **Wih = (double **)calloc(LD, sizeof(double *));
    double **Whh = (double **)calloc(LD, sizeof(double *));
    double **bih = (double **)calloc(LD, sizeof(double *));
    double **bhh = (double **)calloc(LD, sizeof(double *));
    double **Whr = (double **)calloc(LD, sizeof(double *));
    for (int i = 0; i < LD; ++i) {
        const int in_w = i / D == 0 ? in_dim : DHo;
        off_ih[i + 1] = off_ih[i] + (size_t)G * in_w;
        Wih[i] = widen(w[i].w_ih, (size_t)G * in_w, bf16_weights);
        Whh[i] = widen(w[i].w_hh, (size_t)G * Ho, bf16_weights);
        /* biases stay fp32 on both paths */
        bih[i] = widen(w[i].b_ih, (size_t)G, 0);
        bhh[i] = widen(w[i].b_hh, (size_t)G, 0);
        Whr[i] = P > 0 ? widen(w[i].w_hr, (size_t)P * H, bf16_weights) : NULL;
    }
    const int wmax = in_dim > DHo ? in_dim : DHo;
    int nth = 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    nth = omp_get_max_threads();
#endif
    /* per-thread weight-gradient accumulators, summed in thread order at the end */
    const size_t n_ih = off_ih[LD], n_hh = (size_t)LD * G * Ho, n_b = (size_t)LD * G,
                 n_hr = (size_t)LD * P * H;
    const size_t nw = n_ih + n_hh + 2 * n_b + n_hr;
    double *acc = (double *)calloc((size_t)nth * nw, sizeof(double));
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *gWih = acc + (size_t)tid * nw;
        double *gWhh = gWih + n_ih;
        double *gbih = gWhh + n_hh;
        double *gbhh = gbih + n_b;
        double *gWhr = gbhh + n_b;
        /* per row: every layer's input sequence [T][wmax]; per (layer, dir) and
           processing step s: h (s = -1 .. T-1), c, m, gates */
        double *X = (double *)malloc((size_t)layers * T * wmax * sizeof(double));
        double *hs = (double *)malloc((size_t)LD * (T + 1) * Ho * sizeof(double));
        double *cs = (double *)malloc((size_t)LD * (T + 1) * H * sizeof(double));
        double *ms = (double *)malloc((size_t)LD * T * H * sizeof(double));
        double *gt = (double *)malloc((size_t)LD * T * (G + H) * sizeof(double));
        /* clipping: the unclamped cell state and projection of every step */
        double *craw = (double *)malloc((size_t)LD * T * H * sizeof(double));
        double *hraw = (double *)malloc((size_t)LD * T * (P > 0 ? P : 1) * sizeof(double));
        double *dX = (double *)malloc((size_t)T * wmax * sizeof(double));
        double *dY = (double *)malloc((size_t)T * DHo * sizeof(double));
        double *dh = (double *)malloc((size_t)Ho * sizeof(double));
        double *dm = (double *)malloc((size_t)H * sizeof(double));
        double *dc = (double *)malloc((size_t)H * sizeof(double));
        double *dhp = (double *)malloc((size_t)Ho * sizeof(double));
        double *dA = (double *)malloc((size_t)G * sizeof(double));
        double *dR = (double *)malloc((size_t)G * sizeof(double));
        double *pre = (double *)malloc((size_t)2 * G * sizeof(double));
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int b = 0; b < B; ++b) {
            /* row b runs steps t < len (the backward direction from t = len-1) */
            const int len = lengths ? lengths[b] : T;
            /* ---- forward, keeping what the backward needs */
            for (int t = 0; t < T; ++t)
                for (int k = 0; k < in_dim; ++k)
                    X[(size_t)t * wmax + k] = (double)x[((size_t)t * B + b) * in_dim + k];
            for (int l = 0; l < layers; ++l) {
                const int in_w = l == 0 ? in_dim : DHo;
                const double *Xl = X + (size_t)l * T * wmax;
                for (int d = 0; d < D; ++d) {
                    const int i = l * D + d;
                    double *hl = hs + (size_t)i * (T + 1) * Ho, *cl = cs + (size_t)i * (T + 1) * H;
                    double *ml = ms + (size_t)i * T * H;
                    double *gl = gt + (size_t)i * T * (G + H);
                    double *crl = craw + (size_t)i * T * H;
                    double *hrl = hraw + (size_t)i * T * (P > 0 ? P : 1);
                    for (int k = 0; k < Ho; ++k) hl[k] = h0 ? (double)h0[((size_t)i * B + b) * Ho + k] : 0.0;
                    for (int k = 0; k < H; ++k)
                        cl[k] = (lstm && c0) ? (double)c0[((size_t)i * B + b) * H + k] : 0.0;
                    for (int s2 = 0; s2 < len; ++s2) {
                        const int t = d == 0 ? s2 : len - 1 - s2;
                        const double *xt = Xl + (size_t)t * wmax, *hp = hl + (size_t)s2 * Ho;
                        double *hn_ = hl + (size_t)(s2 + 1) * Ho, *cn_ = cl + (size_t)(s2 + 1) * H;
                        double *mt = ml + (size_t)s2 * H;
                        double *g = gl + (size_t)s2 * (G + H);
                        for (int n = 0; n < G; ++n) {
                            double a = bih[i][n], r = bhh[i][n];
                            for (int k = 0; k < in_w; ++k) a += Wih[i][(size_t)n * in_w + k] * xt[k];
                            for (int k = 0; k < Ho; ++k) r += Whh[i][(size_t)n * Ho + k] * hp[k];
                            pre[n] = a;
                            pre[G + n] = r;
                        }
                        for (int u = 0; u < H; ++u) {
                            if (lstm) {
                                const double ig = sigmoid(pre[u] + pre[G + u]);
                                const double f = sigmoid(pre[H + u] + pre[G + H + u]);
                                const double gg = tanh(pre[2 * H + u] + pre[G + 2 * H + u]);
                                const double o = sigmoid(pre[3 * H + u] + pre[G + 3 * H + u]);
                                cn_[u] = f * cl[(size_t)s2 * H + u] + ig * gg;
                                crl[(size_t)s2 * H + u] = cn_[u];
                                if (clip) cn_[u] = clampd(cn_[u], clip[0], clip[1]);
                                mt[u] = o * tanh(cn_[u]);
                                g[u] = ig; g[H + u] = f; g[2 * H + u] = gg; g[3 * H + u] = o;
                            } else {
                                const double r = sigmoid(pre[u] + pre[G + u]);
                                const double z = sigmoid(pre[H + u] + pre[G + H + u]);
                                const double hnp = pre[G + 2 * H + u];  /* W_hn h' + b_hn */
                                const double n = tanh(pre[2 * H + u] + r * hnp);
                                mt[u] = (1.0 - z) * n + z * hp[u];
                                cn_[u] = 0.0;
                                g[u] = r; g[H + u] = z; g[2 * H + u] = n; g[G + u] = hnp;
                            }
                        }
                        if (P > 0) {
                            for (int q = 0; q < P; ++q) {
                                double a2 = 0.0;
                                for (int k = 0; k < H; ++k) a2 += Whr[i][(size_t)q * H + k] * mt[k];
                                hrl[(size_t)s2 * P + q] = a2;
                                hn_[q] = clip ? clampd(a2, clip[2], clip[3]) : a2;
                            }
                        } else {
                            memcpy(hn_, mt, (size_t)H * sizeof(double));
                        }
                        if (l + 1 < layers)  /* next layer input at time t: [h_fwd || h_bwd] */
                            memcpy(X + ((size_t)(l + 1) * T + t) * wmax + (size_t)d * Ho, hn_,
                                   (size_t)Ho * sizeof(double));
                    }
                }
            }
            /* ---- backward, top layer first; direction d replays its steps in reverse */
            for (int t = 0; t < T; ++t)
                for (int k = 0; k < DHo; ++k) dY[(size_t)t * DHo + k] = (double)dy[((size_t)t * B + b) * DHo + k];
            for (int l = layers - 1; l >= 0; --l) {
                const int in_w = l == 0 ? in_dim : DHo;
                const double *Xl = X + (size_t)l * T * wmax;
                for (size_t e = 0; e < (size_t)T * wmax; ++e) dX[e] = 0.0;
                for (int d = 0; d < D; ++d) {
                    const int i = l * D + d;
                    const double *hl = hs + (size_t)i * (T + 1) * Ho, *cl = cs + (size_t)i * (T + 1) * H;
                    const double *ml = ms + (size_t)i * T * H;
                    const double *gl = gt + (size_t)i * T * (G + H);
                    const double *crl = craw + (size_t)i * T * H;
                    const double *hrl = hraw + (size_t)i * T * (P > 0 ? P : 1);
                    for (int k = 0; k < Ho; ++k) dhp[k] = dh_n ? (double)dh_n[((size_t)i * B + b) * Ho + k] : 0.0;
                    for (int k = 0; k < H; ++k)
                        dc[k] = (lstm && dc_n) ? (double)dc_n[((size_t)i * B + b) * H + k] : 0.0;
                    for (int s2 = len - 1; s2 >= 0; --s2) {
                        const int t = d == 0 ? s2 : len - 1 - s2;
                        const double *g = gl + (size_t)s2 * (G + H);
                        const double *hp = hl + (size_t)s2 * Ho, *xt = Xl + (size_t)t * wmax;
                        const double *mt = ml + (size_t)s2 * H;
                        for (int q = 0; q < Ho; ++q) dh[q] = dY[(size_t)t * DHo + (size_t)d * Ho + q] + dhp[q];
                        if (P > 0 && clip)  /* through the projection clamp */
                            for (int q = 0; q < P; ++q) {
                                const double v = hrl[(size_t)s2 * P + q];
                                if (v < clip[2] || v > clip[3]) dh[q] = 0.0;
                            }
                        if (P > 0) {
                            double *gWr = gWhr + (size_t)i * P * H;
                            for (int k = 0; k < H; ++k) {
                                double a2 = 0.0;
                                for (int q = 0; q < P; ++q) a2 += Whr[i][(size_t)q * H + k] * dh[q];
                                dm[k] = a2;
                            }
                            for (int q = 0; q < P; ++q)
                                for (int k = 0; k < H; ++k) gWr[(size_t)q * H + k] += dh[q] * mt[k];
                        } else {
                            memcpy(dm, dh, (size_t)H * sizeof(double));
                        }
                        for (int u = 0; u < H; ++u) {
                            if (lstm) {
                                const double ig = g[u], f = g[H + u], gg = g[2 * H + u], o = g[3 * H + u];
                                const double c = cl[(size_t)(s2 + 1) * H + u], cp = cl[(size_t)s2 * H + u];
                                const double tc = tanh(c);
                                double dcu = dc[u] + dm[u] * o * (1.0 - tc * tc);
                                if (clip) {  /* through the cell-state clamp */
                                    const double v = crl[(size_t)s2 * H + u];
                                    if (v < clip[0] || v > clip[1]) dcu = 0.0;
                                }
                                dA[u] = dcu * gg * ig * (1.0 - ig);
                                dA[H + u] = dcu * cp * f * (1.0 - f);
                                dA[2 * H + u] = dcu * ig * (1.0 - gg * gg);
                                dA[3 * H + u] = dm[u] * tc * o * (1.0 - o);
                                dc[u] = dcu * f;
                                dR[u] = dA[u]; dR[H + u] = dA[H + u];
                                dR[2 * H + u] = dA[2 * H + u]; dR[3 * H + u] = dA[3 * H + u];
                            } else {
                                const double r = g[u], z = g[H + u], n = g[2 * H + u], hnp = g[G + u];
                                const double dn = dm[u] * (1.0 - z);
                                const double dz = dm[u] * (hp[u] - n);
                                const double dan = dn * (1.0 - n * n);
                                const double dr = dan * hnp;
                                dA[u] = dr * r * (1.0 - r);
                                dA[H + u] = dz * z * (1.0 - z);
                                dA[2 * H + u] = dan;
                                dR[u] = dA[u]; dR[H + u] = dA[H + u];
                                dR[2 * H + u] = dan * r;
                            }
                        }
                        /* gradients of this step's weights, input and previous state */
                        double *gWi = gWih + off_ih[i], *gWh = gWhh + (size_t)i * G * Ho;
                        for (int n = 0; n < G; ++n) {
                            for (int k = 0; k < in_w; ++k) gWi[(size_t)n * in_w + k] += dA[n] * xt[k];
                            for (int k = 0; k < Ho; ++k) gWh[(size_t)n * Ho + k] += dR[n] * hp[k];
                            gbih[(size_t)i * G + n] += dA[n];
                            gbhh[(size_t)i * G + n] += dR[n];
                        }
                        for (int k = 0; k < in_w; ++k) {
                            double a2 = 0.0;
                            for (int n = 0; n < G; ++n) a2 += Wih[i][(size_t)n * in_w + k] * dA[n];
                            dX[(size_t)t * wmax + k] += a2;
                        }
                        for (int k = 0; k < Ho; ++k) {
                            double a2 = lstm ? 0.0 : dm[k] * g[H + k];  /* GRU: direct path z h' */
                            for (int n = 0; n < G; ++n) a2 += Whh[i][(size_t)n * Ho + k] * dR[n];
                            dhp[k] = a2;
                        }
                    }
                    for (int k = 0; k < Ho; ++k)
                        if (dh0) dh0[((size_t)i * B + b) * Ho + k] = dhp[k];
                    for (int k = 0; k < H; ++k)
                        if (dc0 && lstm) dc0[((size_t)i * B + b) * H + k] = dc[k];
                }
                if (l > 0) {
                    for (int t = 0; t < T; ++t)
                        memcpy(dY + (size_t)t * DHo, dX + (size_t)t * wmax, (size_t)DHo * sizeof(double));
                } else if (dx) {
                    for (int t = 0; t < T; ++t)
                        for (int k = 0; k < in_dim; ++k)
                            dx[((size_t)t * B + b) * in_dim + k] = dX[(size_t)t * wmax + k];
                }
            }
        }
        free(X); free(hs); free(cs); free(ms); free(gt); free(craw); free(hraw); free(dX); free(dY);
        free(dh); free(dm); free(dc); free(dhp); free(dA); free(dR); free(pre);
    }
    /* sum the per-thread accumulators in thread order */
    double *outs[5] = {dW_ih, dW_hh, db_ih, db_hh, dW_hr};
    const size_t lens[5] = {n_ih, n_hh, n_b, n_b, n_hr};
    size_t base = 0;
    for (int j = 0; j < 5; ++j) {
        if (outs[j])
            for (size_t e = 0; e < lens[j]; ++e) {
                double a2 = 0.0;
                for (int q = 0; q < nth; ++q) a2 += acc[(size_t)q * nw + base + e];
                outs[j][e] = a2;
            }
        base += lens[j];
    }
    free(acc);
    for (int i = 0; i < LD; ++i) {
        free(Wih[i]); free(Whh[i]); free(bih[i]); free(bhh[i]); free(Whr[i]);
    }
    free(Wih); free(Whh); free(bih); free(bhh); free(Whr); free(off_ih);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Backward pass through time of the RSSM prior unroll with given actions   */
/* (the training use of the unroll named in "[Feature Request] CUDNN version */
/* of RSSM", pytorch/rl issue 366, Motivation; the forward is the same       */
/* issue's Solution, as in oracle_rssm_unroll2 above).                       */
/*                                                                          */
/* Given the gradient of a loss with respect to every output of the unroll  */
/* (dmeans, dstds, dstates [T,B,S], dbeliefs [T,B,RH]; any may be NULL =    */
/* 0), returns the gradient with respect to state0 [B,S], belief0 [B,RH],   */
/* the actions [T,B,A] and every weight and bias (summed over rows and      */
/* steps, the weights' own layouts).  The noise eps is an input, not a      */
/* parameter.  One step of the prior, per row, is                            */
/*   u = W1 [s_{t-1}, a_t] + b1,  x = ELU(u)                                 */
/*   h_t = GRUCell(x, h_{t-1})    (r, z, n gates; reset after W_hn h)       */
/*   v = W2 h_t + b2,  q = ELU(v),  p = W3 q + b3                            */
/*   mean = p[0:S],  std = softplus(p[S:2S]) + 0.1,  s_t = mean + eps * std */
/* and the chain rule through these, taken in reverse time, is written out  */
/* term by term below.  Rows are processed one after another (the weight   */
/* gradients sum over all of them).                                          */
/*                                                                          */
/* oracle_rssm_backward2 is the same for the second unroll variant (the     */
/* same issue's Solution, actions computed on the fly): with an actor       */
/* (Wa1 non-NULL) the action of step t is                                    */
/*   a_t = tanh(Wa2 ELU(Wa1 [s_{t-1}, h_{t-1}] + ba1) + ba2)                 */
/* as in oracle_rssm_unroll2, `actions` is not read, dactions[t] is the     */
/* gradient reaching a_t, and the actor's gradients dWa1 [Ha, S+RH], dba1,  */
/* dWa2 [A, Ha], dba2 are returned; its input path adds to the gradients   */
/* of s_{t-1} and h_{t-1}.                                                   */
/* ---------------------------------------------------------------------- */
static double elu_grad(double u) { return u > 0.0 ? 1.0 : exp(u); }

int oracle_rssm_backward2(int S, int A, int Hd, int RH, int T, int B, const float *W1,
                          const float *b1, const float *Wih, const float *Whh, const float *bih,
                          const float *bhh, const float *W2, const float *b2, const float *W3,
                          const float *b3, const float *state0, const float *belief0,
                          const float *actions, const float *eps, const float *dmeans,
                          const float *dstds, const float *dstates, const float *dbeliefs,
                          double *dstate0, double *dbelief0, double *dactions, double *dW1,
                          double *db1, double *dWih, double *dWhh, double *dbih, double *dbhh,
                          double *dW2, double *db2, double *dW3, double *db3, int Ha,
                          const float *Wa1, const float *ba1, const float *Wa2, const float *ba2,
                          double *dWa1, double *dba1, double *dWa2, double *dba2) {
    if (S < 1 || A < 0 || Hd < 1 || RH < 1 || T < 0 || B < 0) return -1;
    const int actor = Wa1 != NULL;
    if (actor && (Ha < 1 || !Wa2 || A < 1 || !dWa1 || !dba1 || !dWa2 || !dba2)) return -1;
    if ((!actor && A > 0 && !actions) || !eps) return -1;
    const int SA = S + A, G = 3 * RH, SR = S + RH;
    const int Hn = actor ? Ha : 1;
    double *wa1 = actor ? widen(Wa1, (size_t)Ha * SR, 0) : NULL;
    double *vba1 = actor ? widen(ba1, Ha, 0) : NULL;
    double *wa2 = actor ? widen(Wa2, (size_t)A * Ha, 0) : NULL;
    double *vba2 = actor ? widen(ba2, A, 0) : NULL;
    if (actor) {
        memset(dWa1, 0, (size_t)Ha * SR * sizeof(double));
        memset(dba1, 0, (size_t)Ha * sizeof(double));
        memset(dWa2, 0, (size_t)A * Ha * sizeof(double));
        memset(dba2, 0, (size_t)A * sizeof(double));
    }
    double *w1 = widen(W1, (size_t)Hd * SA, 0), *vb1 = widen(b1, Hd, 0);
    double *wih = widen(Wih, (size_t)G * Hd, 0), *whh = widen(Whh, (size_t)G * RH, 0);
    double *vbih = widen(bih, G, 0), *vbhh = widen(bhh, G, 0);
    double *w2 = widen(W2, (size_t)Hd * RH, 0), *vb2 = widen(b2, Hd, 0);
    double *w3 = widen(W3, (size_t)2 * S * Hd, 0), *vb3 = widen(b3, (size_t)2 * S, 0);
    memset(dW1, 0, (size_t)Hd * SA * sizeof(double));
    memset(db1, 0, (size_t)Hd * sizeof(double));
    memset(dWih, 0, (size_t)G * Hd * sizeof(double));
    memset(dWhh, 0, (size_t)G * RH * sizeof(double));
    memset(dbih, 0, (size_t)G * sizeof(double));
    memset(dbhh, 0, (size_t)G * sizeof(double));
    memset(dW2, 0, (size_t)Hd * RH * sizeof(double));
    memset(db2, 0, (size_t)Hd * sizeof(double));
    memset(dW3, 0, (size_t)2 * S * Hd * sizeof(double));
    memset(db3, 0, (size_t)2 * S * sizeof(double));
    /* per-step values of one row, kept by the forward for the reverse sweep */
    const size_t Tn = T > 0 ? (size_t)T : 1;
    double *in_s = (double *)calloc(Tn * SA, sizeof(double));   /* [s_{t-1}, a_t] */
    double *u_s = (double *)calloc(Tn * Hd, sizeof(double));
    double *x_s = (double *)calloc(Tn * Hd, sizeof(double));
    double *hp_s = (double *)calloc(Tn * RH, sizeof(double));   /* h_{t-1} */
    double *g_s = (double *)calloc(Tn * G, sizeof(double));     /* r, z, n */
    double *hn_s = (double *)calloc(Tn * RH, sizeof(double));   /* W_hn h_{t-1} + b_hn */
    double *h_s = (double *)calloc(Tn * RH, sizeof(double));
    double *v_s = (double *)calloc(Tn * Hd, sizeof(double));
    double *q_s = (double *)calloc(Tn * Hd, sizeof(double));
    double *p_s = (double *)calloc(Tn * 2 * S, sizeof(double));
    double *ua_s = (double *)calloc(Tn * Hn, sizeof(double));   /* actor pre-ELU */
    double *ha_s = (double *)calloc(Tn * Hn, sizeof(double));   /* actor hidden layer */
    double *dha = (double *)calloc((size_t)Hn, sizeof(double));
    double *dva = (double *)calloc((size_t)(A > 0 ? A : 1), sizeof(double));
    double *gs = (double *)calloc((size_t)S, sizeof(double));    /* dL/ds_t from step t+1 */
    double *gh = (double *)calloc((size_t)RH, sizeof(double));   /* dL/dh_t from step t+1 */
    double *ngs = (double *)calloc((size_t)S, sizeof(double));
    double *ngh = (double *)calloc((size_t)RH, sizeof(double));
    double *dp = (double *)calloc((size_t)2 * S, sizeof(double));
    double *dv = (double *)calloc((size_t)Hd, sizeof(double));
    double *dh = (double *)calloc((size_t)RH, sizeof(double));
    double *din = (double *)calloc((size_t)G, sizeof(double));  /* input-side pre-activations */
    double *dhid = (double *)calloc((size_t)G, sizeof(double)); /* hidden-side */
    double *du = (double *)calloc((size_t)Hd, sizeof(double));
    double *st = (double *)calloc((size_t)S, sizeof(double));
    double *bel = (double *)calloc((size_t)RH, sizeof(double));
    for (int b = 0; b < B; ++b) {
        /* forward of row b */
        for (int j = 0; j < S; ++j) st[j] = state0 ? (double)state0[(size_t)b * S + j] : 0.0;
        for (int j = 0; j < RH; ++j) bel[j] = belief0 ? (double)belief0[(size_t)b * RH + j] : 0.0;
        for (int t = 0; t < T; ++t) {
            double *in = in_s + (size_t)t * SA;
            for (int j = 0; j < S; ++j) in[j] = st[j];
            if (actor) {
                /* a_t = tanh(Wa2 ELU(Wa1 [s_{t-1}, h_{t-1}] + ba1) + ba2) */
                double *ua = ua_s + (size_t)t * Ha, *ha = ha_s + (size_t)t * Ha;
                for (int i = 0; i < Ha; ++i) {
                    double u = vba1 ? vba1[i] : 0.0;
                    for (int j = 0; j < S; ++j) u += wa1[(size_t)i * SR + j] * st[j];
                    for (int j = 0; j < RH; ++j) u += wa1[(size_t)i * SR + S + j] * bel[j];
                    ua[i] = u;
                    ha[i] = elu(u);
                }
                for (int j = 0; j < A; ++j) {
                    double v = vba2 ? vba2[j] : 0.0;
                    for (int i = 0; i < Ha; ++i) v += wa2[(size_t)j * Ha + i] * ha[i];
                    in[S + j] = tanh(v);
                }
            } else {
                for (int j = 0; j < A; ++j) in[S + j] = (double)actions[((size_t)t * B + b) * A + j];
            }
            for (int i = 0; i < Hd; ++i) {
                double u = vb1 ? vb1[i] : 0.0;
                for (int j = 0; j < SA; ++j) u += w1[(size_t)i * SA + j] * in[j];
                u_s[(size_t)t * Hd + i] = u;
                x_s[(size_t)t * Hd + i] = elu(u);
            }
            const double *x = x_s + (size_t)t * Hd;
            memcpy(hp_s + (size_t)t * RH, bel, (size_t)RH * sizeof(double));
            for (int j = 0; j < RH; ++j) {
                double gi[3], gh3[3];
                for (int q = 0; q < 3; ++q) {
                    const int row = q * RH + j;
                    gi[q] = vbih ? vbih[row] : 0.0;
                    gh3[q] = vbhh ? vbhh[row] : 0.0;
                    for (int k = 0; k < Hd; ++k) gi[q] += wih[(size_t)row * Hd + k] * x[k];
                    for (int k = 0; k < RH; ++k) gh3[q] += whh[(size_t)row * RH + k] * bel[k];
                }
                const double r = sigmoid(gi[0] + gh3[0]), z = sigmoid(gi[1] + gh3[1]);
                const double n = tanh(gi[2] + r * gh3[2]);
                double *g = g_s + (size_t)t * G;
                g[j] = r; g[RH + j] = z; g[2 * RH + j] = n;
                hn_s[(size_t)t * RH + j] = gh3[2];
                h_s[(size_t)t * RH + j] = (1.0 - z) * n + z * bel[j];
            }
            memcpy(bel, h_s + (size_t)t * RH, (size_t)RH * sizeof(double));
            for (int i = 0; i < Hd; ++i) {
                double v = vb2 ? vb2[i] : 0.0;
                for (int k = 0; k < RH; ++k) v += w2[(size_t)i * RH + k] * bel[k];
                v_s[(size_t)t * Hd + i] = v;
                q_s[(size_t)t * Hd + i] = elu(v);
            }
            for (int i = 0; i < 2 * S; ++i) {
                double v = vb3 ? vb3[i] : 0.0;
                for (int k = 0; k < Hd; ++k) v += w3[(size_t)i * Hd + k] * q_s[(size_t)t * Hd + k];
                p_s[(size_t)t * 2 * S + i] = v;
            }
            for (int j = 0; j < S; ++j) {
                const double *p = p_s + (size_t)t * 2 * S;
                st[j] = p[j] + (double)eps[((size_t)t * B + b) * S + j] * (softplus(p[S + j]) + 0.1);
            }
        }
        /* reverse sweep of row b */
        memset(gs, 0, (size_t)S * sizeof(double));
        memset(gh, 0, (size_t)RH * sizeof(double));
        for (int t = T - 1; t >= 0; --t) {
            const size_t o = (size_t)t * B + b;
            const double *p = p_s + (size_t)t * 2 * S;
            /* sample: s = mean + eps * (softplus(p_S) + 0.1) */
            for (int j = 0; j < S; ++j) {
                const double ds = (dstates ? (double)dstates[o * S + j] : 0.0) + gs[j];
                const double dmean = (dmeans ? (double)dmeans[o * S + j] : 0.0) + ds;
                const double dsd = (dstds ? (double)dstds[o * S + j] : 0.0) +
                                   ds * (double)eps[o * S + j];
                dp[j] = dmean;
                dp[S + j] = dsd * sigmoid(p[S + j]);  /* d softplus / dp */
            }
            /* head: p = W3 q + b3, q = ELU(v), v = W2 h + b2 */
            const double *q = q_s + (size_t)t * Hd, *h = h_s + (size_t)t * RH;
            for (int i = 0; i < 2 * S; ++i) {
                db3[i] += dp[i];
                for (int k = 0; k < Hd; ++k) dW3[(size_t)i * Hd + k] += dp[i] * q[k];
            }
            for (int k = 0; k < Hd; ++k) {
                double dq = 0.0;
                for (int i = 0; i < 2 * S; ++i) dq += w3[(size_t)i * Hd + k] * dp[i];
                dv[k] = dq * elu_grad(v_s[(size_t)t * Hd + k]);
            }
            for (int i = 0; i < Hd; ++i) {
                db2[i] += dv[i];
                for (int k = 0; k < RH; ++k) dW2[(size_t)i * RH + k] += dv[i] * h[k];
            }
            for (int k = 0; k < RH; ++k) {
                double a = (dbeliefs ? (double)dbeliefs[o * RH + k] : 0.0) + gh[k];
                for (int i = 0; i < Hd; ++i) a += w2[(size_t)i * RH + k] * dv[i];
                dh[k] = a;
            }
            /* GRU cell: h = (1 - z) n + z h_prev, n = tanh(i_n + r * hn) */
            const double *g = g_s + (size_t)t * G, *hp = hp_s + (size_t)t * RH;
            for (int j = 0; j < RH; ++j) {
                const double r = g[j], z = g[RH + j], n = g[2 * RH + j];
                const double dn = dh[j] * (1.0 - z), dz = dh[j] * (hp[j] - n);
                const double dan = dn * (1.0 - n * n);
                const double dar = dan * hn_s[(size_t)t * RH + j] * r * (1.0 - r);
                const double daz = dz * z * (1.0 - z);
                din[j] = dar; din[RH + j] = daz; din[2 * RH + j] = dan;
                dhid[j] = dar; dhid[RH + j] = daz; dhid[2 * RH + j] = dan * r;
                ngh[j] = dh[j] * z;
            }
            const double *x = x_s + (size_t)t * Hd;
            for (int row = 0; row < G; ++row) {
                dbih[row] += din[row];
                dbhh[row] += dhid[row];
                for (int k = 0; k < Hd; ++k) dWih[(size_t)row * Hd + k] += din[row] * x[k];
                for (int k = 0; k < RH; ++k) dWhh[(size_t)row * RH + k] += dhid[row] * hp[k];
            }
            for (int k = 0; k < RH; ++k)
                for (int row = 0; row < G; ++row) ngh[k] += whh[(size_t)row * RH + k] * dhid[row];
            /* input MLP: x = ELU(u), u = W1 [s_{t-1}, a_t] + b1 */
            for (int k = 0; k < Hd; ++k) {
                double dx = 0.0;
                for (int row = 0; row < G; ++row) dx += wih[(size_t)row * Hd + k] * din[row];
                du[k] = dx * elu_grad(u_s[(size_t)t * Hd + k]);
            }
            const double *in = in_s + (size_t)t * SA;
            for (int i = 0; i < Hd; ++i) {
                db1[i] += du[i];
                for (int j = 0; j < SA; ++j) dW1[(size_t)i * SA + j] += du[i] * in[j];
            }
            for (int j = 0; j < SA; ++j) {
                double a = 0.0;
                for (int i = 0; i < Hd; ++i) a += w1[(size_t)i * SA + j] * du[i];
                if (j < S) ngs[j] = a;
                else {
                    if (dactions) dactions[o * A + (j - S)] = a;
                    /* actor: the action's gradient through tanh */
                    if (actor) dva[j - S] = a * (1.0 - in[j] * in[j]);
                }
            }
            if (actor) {
                /* actor: a = tanh(Wa2 ha + ba2), ha = ELU(ua), ua = Wa1 [s_{t-1}, h_{t-1}] + ba1 */
                const double *ua = ua_s + (size_t)t * Ha, *ha = ha_s + (size_t)t * Ha;
                for (int j = 0; j < A; ++j) {
                    dba2[j] += dva[j];
                    for (int i = 0; i < Ha; ++i) dWa2[(size_t)j * Ha + i] += dva[j] * ha[i];
                }
                for (int i = 0; i < Ha; ++i) {
                    double a = 0.0;
                    for (int j = 0; j < A; ++j) a += wa2[(size_t)j * Ha + i] * dva[j];
                    dha[i] = a * elu_grad(ua[i]);
                }
                for (int i = 0; i < Ha; ++i) {
                    dba1[i] += dha[i];
                    for (int j = 0; j < S; ++j) dWa1[(size_t)i * SR + j] += dha[i] * in[j];
                    for (int j = 0; j < RH; ++j) dWa1[(size_t)i * SR + S + j] += dha[i] * hp[j];
                }
                for (int j = 0; j < S; ++j)
                    for (int i = 0; i < Ha; ++i) ngs[j] += wa1[(size_t)i * SR + j] * dha[i];
                for (int j = 0; j < RH; ++j)
                    for (int i = 0; i < Ha; ++i) ngh[j] += wa1[(size_t)i * SR + S + j] * dha[i];
            }
            memcpy(gs, ngs, (size_t)S * sizeof(double));
            memcpy(gh, ngh, (size_t)RH * sizeof(double));
        }
        if (dstate0) memcpy(dstate0 + (size_t)b * S, gs, (size_t)S * sizeof(double));
        if (dbelief0) memcpy(dbelief0 + (size_t)b * RH, gh, (size_t)RH * sizeof(double));
    }
    free(in_s); free(u_s); free(x_s); free(hp_s); free(g_s); free(hn_s); free(h_s);
    free(v_s); free(q_s); free(p_s); free(gs); free(gh); free(ngs); free(ngh); free(dp);
    free(dv); free(dh); free(din); free(dhid); free(du); free(st); free(bel);
    free(ua_s); free(ha_s); free(dha); free(dva);
    free(w1); free(vb1); free(wih); free(whh); free(vbih); free(vbhh);
    free(w2); free(vb2); free(w3); free(vb3);
    free(wa1); free(vba1); free(wa2); free(vba2);
    return 0;
}

int oracle_rssm_backward(int S, int A, int Hd, int RH, int T, int B, const float *W1,
                         const float *b1, const float *Wih, const float *Whh, const float *bih,
                         const float *bhh, const float *W2, const float *b2, const float *W3,
                         const float *b3, const float *state0, const float *belief0,
                         const float *actions, const float *eps, const float *dmeans,
                         const float *dstds, const float *dstates, const float *dbeliefs,
                         double *dstate0, double *dbelief0, double *dactions, double *dW1,
                         double *db1, double *dWih, double *dWhh, double *dbih, double *dbhh,
                         double *dW2, double *db2, double *dW3, double *db3) {
    return oracle_rssm_backward2(S, A, Hd, RH, T, B, W1, b1, Wih, Whh, bih, bhh, W2, b2, W3, b3,
                                 state0, belief0, actions, eps, dmeans, dstds, dstates, dbeliefs,
                                 dstate0, dbelief0, dactions, dW1, db1, dWih, dWhh, dbih, dbhh,
                                 dW2, db2, dW3, db3, 0, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                                 NULL);
}
