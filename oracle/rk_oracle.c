/*
 * rk_oracle.c -- plain, slow, single-threaded CPU oracle of the forward pass
 * of an ONNX recurrent layer (LSTM, GRU, RNN), in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file.  It shares no code, header,
 * table or constant with the CUDA library; the CUDA path never calls it.
 *
 * What it follows (web page "Recurrent layers", onegpu docs):
 *   - section "How a layer runs", step 1: the input projection Xw = X . W^T
 *     of every step and every direction is formed first (rko_projection);
 *   - step 2: the first hidden and cell state come from initial_h /
 *     initial_c, or are zero;
 *   - step 3: one step after another, in order, per direction and batch row;
 *   - step 4: Y in the requested layout, zero past the sequence length;
 *   - section "Arithmetic and determinism": pre = ((xw + rec) + Wb) + Rb,
 *     then the peephole terms (i and f with the previous cell state, o with
 *     the new one), then clip, then the activation, then c = f*c + i*c~,
 *     h = o*h_act(c); GRU h = (1 - z)*h~ + z*h;
 *   - section "Semantics": sequence_lens, Seq = 0, clip with NaN passing
 *     through, input_forget (f = 1 - i), linear_before_reset = 1
 *     (h~ = g(xw_h + r*(rec_h + Rb_h) + Wb_h));
 *   - first paragraph and the C# example: tensors used as stored, W
 *     [dirs, gates*hidden, input], gate order i, o, f, c (LSTM), z, r, h (GRU).
 * The activation formulas are not printed on the pages (they only name the
 * eleven ONNX activations); this file takes them from the ONNX operator
 * definitions.
 *
 * Every value is double.  Half inputs are widened exactly by the caller.
 * No blocking, no fusion, no reordering: sums run in increasing index order.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

/* Oracle-local codes.  The Python wrapper in this folder maps names to them. */
enum { RKO_LSTM = 0, RKO_GRU = 1, RKO_RNN = 2 };
enum { RKO_FORWARD = 0, RKO_REVERSE = 1, RKO_BIDIRECTIONAL = 2 };
enum {
  RKO_SIGMOID = 0, RKO_TANH, RKO_RELU, RKO_AFFINE, RKO_LEAKY_RELU,
  RKO_THRESHOLDED_RELU, RKO_SCALED_TANH, RKO_HARD_SIGMOID, RKO_ELU,
  RKO_SOFTSIGN, RKO_SOFTPLUS
};

typedef struct {
  int32_t cell, direction, layout;
  int64_t seq, batch, input, hidden;
  double clip;               /* <= 0 or NaN: no clip */
  int32_t input_forget;      /* LSTM only */
  int32_t linear_before_reset; /* GRU only */
  int32_t act_kind[6];       /* per direction: LSTM f,g,h; GRU f,g; RNN f */
  double act_alpha[6], act_beta[6];
} rko_problem;

/* ONNX activation functions (the pages name them; the formulas are ONNX's). */
double rko_activation(int32_t kind, double alpha, double beta, double x) {
  switch (kind) {
    case RKO_SIGMOID: return 1.0 / (1.0 + exp(-x));
    case RKO_TANH: return tanh(x);
    case RKO_RELU: return x > 0.0 ? x : (x <= 0.0 ? 0.0 : x); /* NaN stays */
    case RKO_AFFINE: return alpha * x + beta;
    case RKO_LEAKY_RELU: return x >= 0.0 ? x : (x < 0.0 ? alpha * x : x);
    case RKO_THRESHOLDED_RELU: return x > alpha ? x : (x <= alpha ? 0.0 : x);
    case RKO_SCALED_TANH: return alpha * tanh(beta * x);
    case RKO_HARD_SIGMOID: {
      double y = alpha * x + beta;
      if (y < 0.0) return 0.0;
      if (y > 1.0) return 1.0;
      return y;
    }
    case RKO_ELU: return x >= 0.0 ? x : (x < 0.0 ? alpha * (exp(x) - 1.0) : x);
    case RKO_SOFTSIGN: return x / (1.0 + fabs(x));
    case RKO_SOFTPLUS: return log(1.0 + exp(x));
    default: return NAN;
  }
}

/* clip: clamp to [-clip, clip] when clip > 0.  Written as comparisons so a
 * NaN pre-activation passes through ("Semantics": NaN passes through). */
static double rko_clip(double clip, double x) {
  if (!(clip > 0.0)) return x;
  if (x > clip) return clip;
  if (x < -clip) return -clip;
  return x;
}

/* Step 1 of "How a layer runs": the batched Gemm Xw[d] = X . W[d]^T with W
 * in the transposed-B form.  X is [M, K] row-major, W is [D, N, K] row-major,
 * Xw is [D, M, N].  Plain sum in increasing k. */
void rko_projection(int64_t D, int64_t M, int64_t N, int64_t K,
                    const double* X, const double* W, double* Xw) {
  for (int64_t d = 0; d < D; ++d)
    for (int64_t m = 0; m < M; ++m)
      for (int64_t n = 0; n < N; ++n) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
          s += X[m * K + k] * W[(d * N + n) * K + k];
        Xw[(d * M + m) * N + n] = s;
      }
}

static int64_t gates_of(int32_t cell) {
  return cell == RKO_LSTM ? 4 : (cell == RKO_GRU ? 3 : 1);
}
static int64_t acts_per_dir(int32_t cell) {
  return cell == RKO_LSTM ? 3 : (cell == RKO_GRU ? 2 : 1);
}

/* Index helpers for the two layouts ("How a layer runs", step 4; layout 0
 * is [seq, dirs, batch, hidden] for Y and [dirs, batch, hidden] for the
 * states; layout 1 puts batch first). */
static int64_t x_row(const rko_problem* p, int64_t t, int64_t b) {
  return p->layout == 0 ? t * p->batch + b : b * p->seq + t;
}
static int64_t y_off(const rko_problem* p, int64_t D, int64_t t, int64_t d, int64_t b) {
  const int64_t H = p->hidden;
  return p->layout == 0 ? ((t * D + d) * p->batch + b) * H
                        : ((b * p->seq + t) * D + d) * H;
}
static int64_t st_off(const rko_problem* p, int64_t D, int64_t d, int64_t b) {
  const int64_t H = p->hidden;
  return p->layout == 0 ? (d * p->batch + b) * H : (b * D + d) * H;
}

/*
 * The whole layer.  Null inputs mean: B zero, sequence_lens all = seq,
 * initial_h / initial_c zero, P zero.  Null outputs are not written.
 * Shapes (D = 2 for bidirectional, else 1; G gates):
 *   X [seq, batch, input] (layout 0) or [batch, seq, input] (layout 1)
 *   W [D, G*H, input], R [D, G*H, H], B [D, 2*G*H], P [D, 3*H] (i, o, f)
 *   initial_h / initial_c / Y_h / Y_c [D, batch, H] or [batch, D, H]
 *   Y [seq, D, batch, H] or [batch, seq, D, H]
 * Returns 0, or -1 when scratch memory cannot be had.
 */
int rko_layer(const rko_problem* p, const double* X, const double* W,
              const double* R, const double* Bias, const int32_t* seq_lens,
              const double* init_h, const double* init_c, const double* P,
              double* Y, double* Y_h, double* Y_c) {
  const int64_t S = p->seq, NB = p->batch, I = p->input, H = p->hidden;
  const int64_t G = gates_of(p->cell);
  const int64_t D = p->direction == RKO_BIDIRECTIONAL ? 2 : 1;
  const int64_t A = acts_per_dir(p->cell);
  const int is_lstm = p->cell == RKO_LSTM, is_gru = p->cell == RKO_GRU;
  if (NB == 0) return 0;

  double* Xw = NULL;
  if (S > 0 && G * H > 0) {
    Xw = (double*)malloc(sizeof(double) * (size_t)(D * S * NB * G * H));
    if (!Xw) return -1;
    rko_projection(D, S * NB, G * H, I, X, W, Xw);
  }
  double* h = (double*)calloc((size_t)(H > 0 ? H : 1), sizeof(double));
  double* c = (double*)calloc((size_t)(H > 0 ? H : 1), sizeof(double));
  double* hn = (double*)calloc((size_t)(H > 0 ? H : 1), sizeof(double));
  double* zg = (double*)calloc((size_t)(H > 0 ? H : 1), sizeof(double));
  double* rg = (double*)calloc((size_t)(H > 0 ? H : 1), sizeof(double));
  double* pre = (double*)calloc((size_t)(G * H > 0 ? G * H : 1), sizeof(double));
  if (!h || !c || !hn || !zg || !rg || !pre) {
    free(Xw); free(h); free(c); free(hn); free(zg); free(rg); free(pre);
    return -1;
  }

  for (int64_t d = 0; d < D; ++d) {
    const int reverse = p->direction == RKO_REVERSE ||
                        (p->direction == RKO_BIDIRECTIONAL && d == 1);
    const double* Wb = Bias ? Bias + d * 2 * G * H : NULL;
    const double* Rb = Bias ? Bias + d * 2 * G * H + G * H : NULL;
    const double* Rd = R + d * G * H * H;
    const double* Pd = P ? P + d * 3 * H : NULL;
    const int32_t* k = p->act_kind + d * A;
    const double* al = p->act_alpha + d * A;
    const double* be = p->act_beta + d * A;

    for (int64_t b = 0; b < NB; ++b) {
      int64_t L = S;
      if (seq_lens) {
        L = seq_lens[b];
        if (L < 0) L = 0;
        if (L > S) L = S;
      }
      /* step 2: state setup */
      for (int64_t j = 0; j < H; ++j) {
        h[j] = init_h ? init_h[st_off(p, D, d, b) + j] : 0.0;
        c[j] = (is_lstm && init_c) ? init_c[st_off(p, D, d, b) + j] : 0.0;
      }
      if (S == 0) { /* Seq = 0: nothing runs; Y_h, Y_c are the initial states */
        for (int64_t j = 0; j < H; ++j) {
          if (Y_h) Y_h[st_off(p, D, d, b) + j] = h[j];
          if (Y_c && is_lstm) Y_c[st_off(p, D, d, b) + j] = c[j];
        }
        continue;
      }
      if (L == 0) { /* length 0: Y zero, Y_h = Y_c = 0 */
        for (int64_t j = 0; j < H; ++j) { h[j] = 0.0; c[j] = 0.0; }
      }
      /* step 3: the steps, forward from 0 or in reverse from L - 1 */
      for (int64_t s = 0; s < L; ++s) {
        const int64_t t = reverse ? L - 1 - s : s;
        const double* xw = Xw + (d * S * NB + x_row(p, t, b)) * G * H;
        /* pre = ((xw + rec) + Wb) + Rb for every gate row, with rec = R . h */
        for (int64_t r = 0; r < G * H; ++r) {
          double rec = 0.0;
          for (int64_t q = 0; q < H; ++q) rec += Rd[r * H + q] * h[q];
          double v = xw[r] + rec;
          v = v + (Wb ? Wb[r] : 0.0);
          v = v + (Rb ? Rb[r] : 0.0);
          pre[r] = v;
        }
        if (is_lstm) {
          /* gate order i, o, f, c; P order i, o, f */
          for (int64_t j = 0; j < H; ++j) {
            double pi = pre[0 * H + j], po = pre[1 * H + j];
            double pf = pre[2 * H + j], pc = pre[3 * H + j];
            if (Pd) {
              pi = pi + Pd[0 * H + j] * c[j];
              pf = pf + Pd[2 * H + j] * c[j];
            }
            double ig = rko_activation(k[0], al[0], be[0], rko_clip(p->clip, pi));
            double fg = p->input_forget
                            ? 1.0 - ig
                            : rko_activation(k[0], al[0], be[0], rko_clip(p->clip, pf));
            double cg = rko_activation(k[1], al[1], be[1], rko_clip(p->clip, pc));
            double cn = fg * c[j] + ig * cg;
            if (Pd) po = po + Pd[1 * H + j] * cn;
            double og = rko_activation(k[0], al[0], be[0], rko_clip(p->clip, po));
            hn[j] = og * rko_activation(k[2], al[2], be[2], cn);
            c[j] = cn;
          }
        } else if (is_gru) {
          /* gate order z, r, h */
          for (int64_t j = 0; j < H; ++j) {
            zg[j] = rko_activation(k[0], al[0], be[0], rko_clip(p->clip, pre[0 * H + j]));
            rg[j] = rko_activation(k[0], al[0], be[0], rko_clip(p->clip, pre[1 * H + j]));
          }
          for (int64_t j = 0; j < H; ++j) {
            double ph;
            const double wbh = Wb ? Wb[2 * H + j] : 0.0;
            const double rbh = Rb ? Rb[2 * H + j] : 0.0;
            if (p->linear_before_reset) {
              /* h~ = g(xw_h + r*(rec_h + Rb_h) + Wb_h), rec_h = R_h . h */
              double rec = 0.0;
              for (int64_t q = 0; q < H; ++q) rec += Rd[(2 * H + j) * H + q] * h[q];
              ph = (xw[2 * H + j] + rg[j] * (rec + rbh)) + wbh;
            } else {
              /* the candidate's product takes r (.) h of every unit */
              double rec = 0.0;
              for (int64_t q = 0; q < H; ++q) rec += Rd[(2 * H + j) * H + q] * (rg[q] * h[q]);
              ph = ((xw[2 * H + j] + rec) + wbh) + rbh;
            }
            double hc = rko_activation(k[1], al[1], be[1], rko_clip(p->clip, ph));
            hn[j] = (1.0 - zg[j]) * hc + zg[j] * h[j];
          }
        } else {
          for (int64_t j = 0; j < H; ++j)
            hn[j] = rko_activation(k[0], al[0], be[0], rko_clip(p->clip, pre[j]));
        }
        for (int64_t j = 0; j < H; ++j) h[j] = hn[j];
        if (Y) for (int64_t j = 0; j < H; ++j) Y[y_off(p, D, t, d, b) + j] = h[j];
      }
      /* step 4: Y is zero at the steps past the length */
      if (Y)
        for (int64_t t = L; t < S; ++t)
          for (int64_t j = 0; j < H; ++j) Y[y_off(p, D, t, d, b) + j] = 0.0;
      for (int64_t j = 0; j < H; ++j) {
        if (Y_h) Y_h[st_off(p, D, d, b) + j] = h[j];
        if (Y_c && is_lstm) Y_c[st_off(p, D, d, b) + j] = c[j];
      }
    }
  }
  free(Xw); free(h); free(c); free(hn); free(zg); free(rg); free(pre);
  return 0;
}
