/*
 * gpt2_oracle.c -- plain, slow, double-precision CPU oracle of the GPT-2
 * forward pass and of its KV-cached decode step.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  It shares no
 * code with the CUDA library: no headers, no helpers, no constants.
 *
 * Every step is written the plain way, from its definition:
 *   - encoder: token embedding plus position embedding ("Encoder" kernel of
 *     the ECE408 GPT-2 project page, grade table);
 *   - LayerNorm over the channel axis, biased variance, eps = 1e-5
 *     ("LayerNorm" kernel, same table; eps and variance form are GPT-2's,
 *     the page is silent on them);
 *   - matmul with bias, y = x W^T + b with W stored [out, in] ("MatMul");
 *   - causal multi-head attention by FlashAttention's Algorithm 0 (the
 *     standard implementation: scores, mask, softmax, times V), heads taken as
 *     column blocks of the fused QKV projection (NanoGPT project, "Head
 *     Splitting and Tensor Shapes"); scale 1/sqrt(head size);
 *   - an independent Algorithm 1 recompute (tiled, online softmax), used
 *     only to cross-check Algorithm 0 (FlashAttention (I), Task 2);
 *   - the backward algorithms of Algorithms 0 and 1 for causal attention
 *     (FlashAttention (II): the chain rule through the softmax, and its
 *     tiled form recomputing the attention matrix from row statistics);
 *   - tanh-form GELU, the residual add, the vocabulary softmax;
 *   - the KV-cached decode step (NanoGPT project, "KV Caching");
 *   - a training step's loss and gradient (softmax cross-entropy and the
 *     backward of every forward step) and AdamW (llm.c "State of the
 *     Union": forward blocks, classifier, backward blocks, optimizer).
 * All arithmetic is in double; parameters arrive as the caller's fp32 buffer
 * and are widened exactly.  OpenMP pragmas only split independent output
 * elements across threads: each element is still summed by one thread in
 * the order written, so results do not depend on the thread count.
 *
 * Parity pins for every function live in the test suite (closed forms,
 * invariants, brute force and library cross-checks); none is unpinned.
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int max_seq_len;        /* maxT */
  int vocab_size;         /* V */
  int padded_vocab_size;  /* Vp */
  int num_layers;         /* L */
  int num_heads;          /* NH */
  int channels;           /* C */
} OracleGPT2Config;

#define ORACLE_LN_EPS 1e-5

/* ---------------------------------------------------------------- encoder */
/* out[b,t,c] = wte[tok[b,t], c] + wpe[t, c] */
void oracle_encoder(double* out, const int* tok, const float* wte, const float* wpe,
                    int B, int T, int C) {
  for (int b = 0; b < B; b++)
    for (int t = 0; t < T; t++) {
      const int ix = tok[b * T + t];
      for (int c = 0; c < C; c++)
        out[((size_t)b * T + t) * C + c] = (double)wte[(size_t)ix * C + c] + (double)wpe[(size_t)t * C + c];
    }
}

/* ------------------------------------------------------------- layernorm */
/* y = (x - mean) / sqrt(var + eps) * w + b over each row of C values.
 * mean and rstd (= 1/sqrt(var+eps)) are returned per row when non-null. */
void oracle_layernorm(double* out, double* mean_out, double* rstd_out, const double* inp,
                      const float* w, const float* bias, int N, int C) {
  for (int n = 0; n < N; n++) {
    const double* x = inp + (size_t)n * C;
    double mean = 0.0;
    for (int c = 0; c < C; c++) mean += x[c];
    mean /= C;
    double var = 0.0;
    for (int c = 0; c < C; c++) var += (x[c] - mean) * (x[c] - mean);
    var /= C;
    const double rstd = 1.0 / sqrt(var + ORACLE_LN_EPS);
    for (int c = 0; c < C; c++)
      out[(size_t)n * C + c] = (x[c] - mean) * rstd * (double)w[c] + (double)bias[c];
    if (mean_out) mean_out[n] = mean;
    if (rstd_out) rstd_out[n] = rstd;
  }
}

/* ---------------------------------------------------------------- matmul */
/* out[n, o] = bias[o] + sum_k inp[n, k] * W[o, k];  W is [OC, C] row-major.
 * bias may be null (the LM head has none). */
void oracle_matmul(double* out, const double* inp, const float* W, const float* bias,
                   int N, int C, int OC) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; n++) {
    const double* x = inp + (size_t)n * C;
    for (int o = 0; o < OC; o++) {
      const float* wrow = W + (size_t)o * C;
      double acc = bias ? (double)bias[o] : 0.0;
      for (int k = 0; k < C; k++) acc += x[k] * (double)wrow[k];
      out[(size_t)n * OC + o] = acc;
    }
  }
}

/* Same with a double-precision weight matrix (used by the single-kernel
 * tests, whose weights are not part of a parameter buffer). */
void oracle_matmul_f64w(double* out, const double* inp, const double* W, const double* bias,
                        int N, int C, int OC) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; n++) {
    const double* x = inp + (size_t)n * C;
    for (int o = 0; o < OC; o++) {
      const double* wrow = W + (size_t)o * C;
      double acc = bias ? bias[o] : 0.0;
      for (int k = 0; k < C; k++) acc += x[k] * wrow[k];
      out[(size_t)n * OC + o] = acc;
    }
  }
}

/* ------------------------------------------------------------- attention */
/* Algorithm 0 (standard attention) for causal multi-head self-attention.
 * qkv is [B, T, 3C]: columns [0,C) are queries, [C,2C) keys, [2C,3C) values;
 * head h owns columns [h*hs, (h+1)*hs) of each block.  out is [B, T, C] with
 * the heads concatenated in the same column order.
 *   S[t, j] = q_t . k_j / sqrt(hs)   for j <= t, -inf for j > t
 *   P = row softmax of S;  out_t = sum_j P[t, j] v_j                        */
void oracle_attention(double* out, const double* qkv, int B, int T, int C, int NH) {
  const int hs = C / NH;
  const double scale = 1.0 / sqrt((double)hs);
#pragma omp parallel for collapse(2) schedule(static)
  for (int b = 0; b < B; b++)
    for (int h = 0; h < NH; h++) {
      double* S = (double*)malloc(sizeof(double) * (size_t)T * T);
      for (int t = 0; t < T; t++) {
        const double* q = qkv + ((size_t)b * T + t) * 3 * C + h * hs;
        for (int j = 0; j < T; j++) {
          if (j > t) { S[(size_t)t * T + j] = -INFINITY; continue; }
          const double* k = qkv + ((size_t)b * T + j) * 3 * C + C + h * hs;
          double dot = 0.0;
          for (int d = 0; d < hs; d++) dot += q[d] * k[d];
          S[(size_t)t * T + j] = dot * scale;
        }
        /* softmax over the row; exp(-inf) = 0 removes the masked entries */
        double mx = -INFINITY;
        for (int j = 0; j < T; j++) if (S[(size_t)t * T + j] > mx) mx = S[(size_t)t * T + j];
        double sum = 0.0;
        for (int j = 0; j < T; j++) {
          S[(size_t)t * T + j] = exp(S[(size_t)t * T + j] - mx);
          sum += S[(size_t)t * T + j];
        }
        for (int j = 0; j < T; j++) S[(size_t)t * T + j] /= sum;
        double* o = out + ((size_t)b * T + t) * C + h * hs;
        for (int d = 0; d < hs; d++) {
          double acc = 0.0;
          for (int j = 0; j < T; j++)
            acc += S[(size_t)t * T + j] * qkv[((size_t)b * T + j) * 3 * C + 2 * C + h * hs + d];
          o[d] = acc;
        }
      }
      free(S);
    }
}

/* Algorithm 1 (FlashAttention forward): queries in blocks of Br rows, keys
 * and values in blocks of Bc rows.  For each query block, running row maxima
 * m, running row sums l and a normalised output O are updated block by block:
 *   S = Q K_j^T * scale (causal mask), mt = rowmax(S), Pt = exp(S - mt),
 *   lt = rowsum(Pt), m_new = max(m, mt),
 *   l_new = exp(m - m_new) l + exp(mt - m_new) lt,
 *   O = (l exp(m - m_new) O + exp(mt - m_new) Pt V_j) / l_new.
 * Key blocks that lie wholly after the query block are skipped.  A row with
 * every key of a block masked takes no update from that block. */
void oracle_attention_online(double* out, const double* qkv, int B, int T, int C, int NH,
                             int Br, int Bc) {
  const int hs = C / NH;
  const double scale = 1.0 / sqrt((double)hs);
  double* S = (double*)malloc(sizeof(double) * (size_t)Br * Bc);
  double* m = (double*)malloc(sizeof(double) * Br);
  double* l = (double*)malloc(sizeof(double) * Br);
  double* O = (double*)malloc(sizeof(double) * (size_t)Br * hs);
  for (int b = 0; b < B; b++)
    for (int h = 0; h < NH; h++)
      for (int i0 = 0; i0 < T; i0 += Br) {
        const int br = (T - i0 < Br) ? T - i0 : Br;
        for (int r = 0; r < br; r++) {
          m[r] = -INFINITY;
          l[r] = 0.0;
          for (int d = 0; d < hs; d++) O[(size_t)r * hs + d] = 0.0;
        }
        for (int j0 = 0; j0 < T; j0 += Bc) {
          if (j0 > i0 + br - 1) break;  /* every key in this block is after every query */
          const int bc = (T - j0 < Bc) ? T - j0 : Bc;
          for (int r = 0; r < br; r++) {
            const int t = i0 + r;
            const double* q = qkv + ((size_t)b * T + t) * 3 * C + h * hs;
            double mt = -INFINITY;
            for (int c = 0; c < bc; c++) {
              const int j = j0 + c;
              double s = -INFINITY;
              if (j <= t) {
                const double* k = qkv + ((size_t)b * T + j) * 3 * C + C + h * hs;
                double dot = 0.0;
                for (int d = 0; d < hs; d++) dot += q[d] * k[d];
                s = dot * scale;
              }
              S[(size_t)r * Bc + c] = s;
              if (s > mt) mt = s;
            }
            if (mt == -INFINITY) continue;  /* row wholly masked in this block */
            double lt = 0.0;
            for (int c = 0; c < bc; c++) {
              S[(size_t)r * Bc + c] = exp(S[(size_t)r * Bc + c] - mt);
              lt += S[(size_t)r * Bc + c];
            }
            const double m_new = (m[r] > mt) ? m[r] : mt;
            const double a_old = exp(m[r] - m_new);  /* exp(-inf) = 0 on the first block */
            const double a_new = exp(mt - m_new);
            const double l_new = a_old * l[r] + a_new * lt;
            for (int d = 0; d < hs; d++) {
              double pv = 0.0;
              for (int c = 0; c < bc; c++)
                pv += S[(size_t)r * Bc + c] * qkv[((size_t)b * T + j0 + c) * 3 * C + 2 * C + h * hs + d];
              O[(size_t)r * hs + d] = (l[r] * a_old * O[(size_t)r * hs + d] + a_new * pv) / l_new;
            }
            m[r] = m_new;
            l[r] = l_new;
          }
        }
        for (int r = 0; r < br; r++)
          for (int d = 0; d < hs; d++)
            out[((size_t)b * T + i0 + r) * C + h * hs + d] = O[(size_t)r * hs + d];
      }
  free(S); free(m); free(l); free(O);
}

/* ------------------------------------------------------ attention backward */
/* The backward pass of causal attention (FlashAttention (II): the backward
 * algorithm of Algorithm 0).  Given dout = dL/dO [B,T,C], per (b, h), with
 * S = Q K^T * scale (masked), P = softmax_rows(S), O = P V:
 *   dV = P^T dO,  dP = dO V^T,
 *   dS[t][j] = P[t][j] (dP[t][j] - sum_k P[t][k] dP[t][k])   (the softmax
 *              Jacobian applied to row t),
 *   dQ = dS K * scale,  dK = dS^T Q * scale.
 * dqkv [B,T,3C] holds dQ, dK, dV in the column blocks of Q, K, V. */
void oracle_attention_backward(double* dqkv, const double* dout, const double* qkv, int B, int T, int C, int NH) {
  const int hs = C / NH;
  const double scale = 1.0 / sqrt((double)hs);
  memset(dqkv, 0, sizeof(double) * (size_t)B * T * 3 * C);
#pragma omp parallel for collapse(2) schedule(static)
  for (int b = 0; b < B; b++)
    for (int h = 0; h < NH; h++) {
      double* P = (double*)malloc(sizeof(double) * (size_t)T * T);
      double* dP = (double*)malloc(sizeof(double) * (size_t)T * T);
      const double* base = qkv + (size_t)b * T * 3 * C;
      double* dbase = dqkv + (size_t)b * T * 3 * C;
      /* P: the forward's probabilities, as in oracle_attention */
      for (int t = 0; t < T; t++) {
        const double* q = base + (size_t)t * 3 * C + h * hs;
        double mx = -INFINITY;
        for (int j = 0; j <= t; j++) {
          const double* k = base + (size_t)j * 3 * C + C + h * hs;
          double dot = 0.0;
          for (int d = 0; d < hs; d++) dot += q[d] * k[d];
          P[(size_t)t * T + j] = dot * scale;
          if (P[(size_t)t * T + j] > mx) mx = P[(size_t)t * T + j];
        }
        double sum = 0.0;
        for (int j = 0; j <= t; j++) {
          P[(size_t)t * T + j] = exp(P[(size_t)t * T + j] - mx);
          sum += P[(size_t)t * T + j];
        }
        for (int j = 0; j <= t; j++) P[(size_t)t * T + j] /= sum;
        for (int j = t + 1; j < T; j++) P[(size_t)t * T + j] = 0.0;
      }
      /* dP = dO V^T (only j <= t matters) and dV = P^T dO */
      for (int t = 0; t < T; t++) {
        const double* go = dout + ((size_t)b * T + t) * C + h * hs;
        for (int j = 0; j <= t; j++) {
          const double* v = base + (size_t)j * 3 * C + 2 * C + h * hs;
          double dot = 0.0;
          for (int d = 0; d < hs; d++) dot += go[d] * v[d];
          dP[(size_t)t * T + j] = dot;
        }
      }
      for (int j = 0; j < T; j++) {
        double* dv = dbase + (size_t)j * 3 * C + 2 * C + h * hs;
        for (int d = 0; d < hs; d++) {
          double acc = 0.0;
          for (int t = j; t < T; t++) acc += P[(size_t)t * T + j] * dout[((size_t)b * T + t) * C + h * hs + d];
          dv[d] = acc;
        }
      }
      /* dS, written over dP */
      for (int t = 0; t < T; t++) {
        double rowdot = 0.0;
        for (int k = 0; k <= t; k++) rowdot += P[(size_t)t * T + k] * dP[(size_t)t * T + k];
        for (int j = 0; j <= t; j++) dP[(size_t)t * T + j] = P[(size_t)t * T + j] * (dP[(size_t)t * T + j] - rowdot);
      }
      /* dQ = dS K * scale, dK = dS^T Q * scale */
      for (int t = 0; t < T; t++) {
        double* dq = dbase + (size_t)t * 3 * C + h * hs;
        for (int d = 0; d < hs; d++) {
          double acc = 0.0;
          for (int j = 0; j <= t; j++) acc += dP[(size_t)t * T + j] * base[(size_t)j * 3 * C + C + h * hs + d];
          dq[d] = acc * scale;
        }
      }
      for (int j = 0; j < T; j++) {
        double* dk = dbase + (size_t)j * 3 * C + C + h * hs;
        for (int d = 0; d < hs; d++) {
          double acc = 0.0;
          for (int t = j; t < T; t++) acc += dP[(size_t)t * T + j] * base[(size_t)t * 3 * C + h * hs + d];
          dk[d] = acc * scale;
        }
      }
      free(P);
      free(dP);
    }
}

/* The backward algorithm of Algorithm 1 (FlashAttention (II)): tiled, with
 * the attention matrix recomputed block by block instead of stored.  The
 * forward leaves per row the statistic L = m + log(l) (its running maximum
 * and sum; P = exp(S - L)), computed here by a first tiled sweep, and
 * D[t] = sum_d dO[t][d] O[t][d] (which equals sum_k P[t][k] dP[t][k]).  Then
 * for each key block j and each query block i that sees it:
 *   P = exp(S_ij - L_i), dV_j += P^T dO_i, dP = dO_i V_j^T,
 *   dS = P (dP - D_i), dQ_i += dS K_j * scale, dK_j += dS^T Q_i * scale.
 * `out` is the forward output O [B,T,C]. */
void oracle_attention_backward_online(double* dqkv, const double* dout, const double* qkv, const double* out,
                                      int B, int T, int C, int NH, int Br, int Bc) {
  const int hs = C / NH;
  const double scale = 1.0 / sqrt((double)hs);
  memset(dqkv, 0, sizeof(double) * (size_t)B * T * 3 * C);
  double* L = (double*)malloc(sizeof(double) * T);
  double* D = (double*)malloc(sizeof(double) * T);
  double* Pt = (double*)malloc(sizeof(double) * (size_t)Br * Bc);
  for (int b = 0; b < B; b++)
    for (int h = 0; h < NH; h++) {
      const double* base = qkv + (size_t)b * T * 3 * C;
      double* dbase = dqkv + (size_t)b * T * 3 * C;
      /* the forward's row statistics, block by block (online max and sum) */
      for (int t = 0; t < T; t++) {
        const double* q = base + (size_t)t * 3 * C + h * hs;
        double m = -INFINITY, l = 0.0;
        for (int j0 = 0; j0 <= t; j0 += Bc) {
          double mt = -INFINITY;
          const int je = (j0 + Bc - 1 < t) ? j0 + Bc - 1 : t;
          for (int j = j0; j <= je; j++) {
            const double* k = base + (size_t)j * 3 * C + C + h * hs;
            double dot = 0.0;
            for (int d = 0; d < hs; d++) dot += q[d] * k[d];
            if (dot * scale > mt) mt = dot * scale;
          }
          const double m_new = m > mt ? m : mt;
          double lt = 0.0;
          for (int j = j0; j <= je; j++) {
            const double* k = base + (size_t)j * 3 * C + C + h * hs;
            double dot = 0.0;
            for (int d = 0; d < hs; d++) dot += q[d] * k[d];
            lt += exp(dot * scale - m_new);
          }
          l = l * exp(m - m_new) + lt;
          m = m_new;
        }
        L[t] = m + log(l);
        double dd = 0.0;
        for (int d = 0; d < hs; d++)
          dd += dout[((size_t)b * T + t) * C + h * hs + d] * out[((size_t)b * T + t) * C + h * hs + d];
        D[t] = dd;
      }
      for (int j0 = 0; j0 < T; j0 += Bc) {
        const int bc = (T - j0 < Bc) ? T - j0 : Bc;
        for (int i0 = (j0 / Br) * Br; i0 < T; i0 += Br) {  /* query blocks that can see key block j0 */
          const int br = (T - i0 < Br) ? T - i0 : Br;
          for (int r = 0; r < br; r++) {
            const int t = i0 + r;
            const double* q = base + (size_t)t * 3 * C + h * hs;
            for (int c = 0; c < bc; c++) {
              const int j = j0 + c;
              double p = 0.0;
              if (j <= t) {
                const double* k = base + (size_t)j * 3 * C + C + h * hs;
                double dot = 0.0;
                for (int d = 0; d < hs; d++) dot += q[d] * k[d];
                p = exp(dot * scale - L[t]);
              }
              Pt[(size_t)r * Bc + c] = p;
            }
          }
          for (int r = 0; r < br; r++) {
            const int t = i0 + r;
            const double* go = dout + ((size_t)b * T + t) * C + h * hs;
            for (int c = 0; c < bc; c++) {
              const int j = j0 + c;
              const double p = Pt[(size_t)r * Bc + c];
              if (p == 0.0) continue;
              const double* v = base + (size_t)j * 3 * C + 2 * C + h * hs;
              double dp = 0.0;
              for (int d = 0; d < hs; d++) dp += go[d] * v[d];
              const double ds = p * (dp - D[t]);
              double* dq = dbase + (size_t)t * 3 * C + h * hs;
              double* dk = dbase + (size_t)j * 3 * C + C + h * hs;
              double* dv = dbase + (size_t)j * 3 * C + 2 * C + h * hs;
              const double* k = base + (size_t)j * 3 * C + C + h * hs;
              const double* q = base + (size_t)t * 3 * C + h * hs;
              for (int d = 0; d < hs; d++) {
                dv[d] += p * go[d];
                dq[d] += ds * k[d] * scale;
                dk[d] += ds * q[d] * scale;
              }
            }
          }
        }
      }
    }
  free(L);
  free(D);
  free(Pt);
}

/* ------------------------------------------------------------ elementwise */
/* GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
void oracle_gelu(double* out, const double* inp, int n) {
  const double s2pi = sqrt(2.0 / M_PI);
  for (int i = 0; i < n; i++) {
    const double x = inp[i];
    out[i] = 0.5 * x * (1.0 + tanh(s2pi * (x + 0.044715 * x * x * x)));
  }
}

/* out = a + b */
void oracle_residual(double* out, const double* a, const double* b, int n) {
  for (int i = 0; i < n; i++) out[i] = a[i] + b[i];
}

/* ---------------------------------------------------------------- softmax */
/* probs[n, v] = exp(l[n,v] - max) / sum_{u<V} exp(l[n,u] - max) for v < V,
 * and 0 for the padded columns V <= v < Vp. */
void oracle_softmax(double* probs, const double* logits, int N, int V, int Vp) {
  for (int n = 0; n < N; n++) {
    const double* lrow = logits + (size_t)n * Vp;
    double* prow = probs + (size_t)n * Vp;
    double mx = -INFINITY;
    for (int v = 0; v < V; v++) if (lrow[v] > mx) mx = lrow[v];
    double sum = 0.0;
    for (int v = 0; v < V; v++) sum += exp(lrow[v] - mx);
    for (int v = 0; v < V; v++) prow[v] = exp(lrow[v] - mx) / sum;
    for (int v = V; v < Vp; v++) prow[v] = 0.0;
  }
}

/* ----------------------------------------------------------------- argmax */
/* next[b] = smallest v < V with the largest logits[b, v] */
void oracle_argmax(int* next, const double* logits, int B, int V, int Vp) {
  for (int b = 0; b < B; b++) {
    int best = 0;
    for (int v = 1; v < V; v++)
      if (logits[(size_t)b * Vp + v] > logits[(size_t)b * Vp + best]) best = v;
    next[b] = best;
  }
}

/* ------------------------------------------------------------- parameters */
typedef struct {
  const float *wte, *wpe, *ln1w, *ln1b, *qkvw, *qkvb, *attprojw, *attprojb,
      *ln2w, *ln2b, *fcw, *fcb, *fcprojw, *fcprojb, *lnfw, *lnfb;
} OracleParams;

/* The flat buffer holds the tensors in this order, each row-major:
 * wte[Vp,C] wpe[maxT,C] ln1w[L,C] ln1b[L,C] qkvw[L,3C,C] qkvb[L,3C]
 * attprojw[L,C,C] attprojb[L,C] ln2w[L,C] ln2b[L,C] fcw[L,4C,C] fcb[L,4C]
 * fcprojw[L,C,4C] fcprojb[L,C] lnfw[C] lnfb[C] */
static OracleParams oracle_params(const OracleGPT2Config* cfg, const float* p) {
  const size_t C = cfg->channels, L = cfg->num_layers, Vp = cfg->padded_vocab_size,
               maxT = cfg->max_seq_len;
  OracleParams w;
  w.wte = p; p += Vp * C;
  w.wpe = p; p += maxT * C;
  w.ln1w = p; p += L * C;
  w.ln1b = p; p += L * C;
  w.qkvw = p; p += L * 3 * C * C;
  w.qkvb = p; p += L * 3 * C;
  w.attprojw = p; p += L * C * C;
  w.attprojb = p; p += L * C;
  w.ln2w = p; p += L * C;
  w.ln2b = p; p += L * C;
  w.fcw = p; p += L * 4 * C * C;
  w.fcb = p; p += L * 4 * C;
  w.fcprojw = p; p += L * 4 * C * C;
  w.fcprojb = p; p += L * C;
  w.lnfw = p; p += C;
  w.lnfb = p; p += C;
  return w;
}

size_t oracle_num_params(const OracleGPT2Config* cfg) {
  const size_t C = cfg->channels, L = cfg->num_layers;
  return (size_t)cfg->padded_vocab_size * C + (size_t)cfg->max_seq_len * C +
         L * (2 * C + 3 * C * C + 3 * C + C * C + C + 2 * C + 4 * C * C + 4 * C + 4 * C * C + C) + 2 * C;
}

/* ----------------------------------------------------- the forward pass */
/* Final hidden state h = LN_f(x_L) for B sequences of T tokens, [B*T, C].
 * When kcache/vcache are non-null (each [L, B, NH, maxT, hs]) the keys and
 * values of every layer are stored there at positions [0, T). */
void oracle_gpt2_hidden(const OracleGPT2Config* cfg, const float* params, const int* tok,
                        int B, int T, double* hidden, double* kcache, double* vcache) {
  const int C = cfg->channels, L = cfg->num_layers, NH = cfg->num_heads, hs = C / NH;
  const int maxT = cfg->max_seq_len;
  const size_t N = (size_t)B * T;
  OracleParams w = oracle_params(cfg, params);
  double* x = (double*)malloc(sizeof(double) * N * C);
  double* h = (double*)malloc(sizeof(double) * N * C);
  double* qkv = (double*)malloc(sizeof(double) * N * 3 * C);
  double* att = (double*)malloc(sizeof(double) * N * C);
  double* proj = (double*)malloc(sizeof(double) * N * C);
  double* fc = (double*)malloc(sizeof(double) * N * 4 * C);
  double* fcg = (double*)malloc(sizeof(double) * N * 4 * C);

  oracle_encoder(x, tok, w.wte, w.wpe, B, T, C);
  for (int l = 0; l < L; l++) {
    /* attention sub-block: x = x + proj(attention(LN1(x))) */
    oracle_layernorm(h, NULL, NULL, x, w.ln1w + (size_t)l * C, w.ln1b + (size_t)l * C, (int)N, C);
    oracle_matmul(qkv, h, w.qkvw + (size_t)l * 3 * C * C, w.qkvb + (size_t)l * 3 * C, (int)N, C, 3 * C);
    if (kcache && vcache)
      for (int b = 0; b < B; b++)
        for (int hd = 0; hd < NH; hd++)
          for (int t = 0; t < T; t++)
            for (int d = 0; d < hs; d++) {
              const size_t ci = ((((size_t)l * B + b) * NH + hd) * maxT + t) * hs + d;
              const size_t qi = ((size_t)b * T + t) * 3 * C + hd * hs + d;
              kcache[ci] = qkv[qi + C];
              vcache[ci] = qkv[qi + 2 * C];
            }
    oracle_attention(att, qkv, B, T, C, NH);
    oracle_matmul(proj, att, w.attprojw + (size_t)l * C * C, w.attprojb + (size_t)l * C, (int)N, C, C);
    oracle_residual(x, x, proj, (int)(N * C));
    /* MLP sub-block: x = x + fcproj(GELU(fc(LN2(x)))) */
    oracle_layernorm(h, NULL, NULL, x, w.ln2w + (size_t)l * C, w.ln2b + (size_t)l * C, (int)N, C);
    oracle_matmul(fc, h, w.fcw + (size_t)l * 4 * C * C, w.fcb + (size_t)l * 4 * C, (int)N, C, 4 * C);
    oracle_gelu(fcg, fc, (int)(N * 4 * C));
    oracle_matmul(proj, fcg, w.fcprojw + (size_t)l * 4 * C * C, w.fcprojb + (size_t)l * C, (int)N, 4 * C, C);
    oracle_residual(x, x, proj, (int)(N * C));
  }
  oracle_layernorm(hidden, NULL, NULL, x, w.lnfw, w.lnfb, (int)N, C);
  free(x); free(h); free(qkv); free(att); free(proj); free(fc); free(fcg);
}

/* LM head, tied to the token embedding and without bias: logits = h wte^T
 * over all Vp rows of wte, for N rows of h. */
void oracle_lm_head(const OracleGPT2Config* cfg, const float* params, const double* hidden,
                    int N, double* logits) {
  OracleParams w = oracle_params(cfg, params);
  oracle_matmul(logits, hidden, w.wte, NULL, N, cfg->channels, cfg->padded_vocab_size);
}

/* The whole forward pass: logits [B*T, Vp] and, when probs is non-null,
 * the vocabulary softmax of each row. */
void oracle_gpt2_forward(const OracleGPT2Config* cfg, const float* params, const int* tok,
                         int B, int T, double* logits, double* probs,
                         double* kcache, double* vcache) {
  const size_t N = (size_t)B * T;
  double* hidden = (double*)malloc(sizeof(double) * N * cfg->channels);
  oracle_gpt2_hidden(cfg, params, tok, B, T, hidden, kcache, vcache);
  oracle_lm_head(cfg, params, hidden, (int)N, logits);
  if (probs) oracle_softmax(probs, logits, (int)N, cfg->vocab_size, cfg->padded_vocab_size);
  free(hidden);
}

/* ---------------------------------------------------- the decode step */
/* One new token per sequence at position pos (0 <= pos < maxT), given the
 * keys and values of positions [0, pos) in kcache/vcache ([L,B,NH,maxT,hs]).
 * Stores this position's keys and values at pos, then attends over [0, pos].
 * The arithmetic per row is the forward pass's, restricted to row pos. */
void oracle_gpt2_decode_step(const OracleGPT2Config* cfg, const float* params,
                             double* kcache, double* vcache, const int* tok, int B, int pos,
                             double* logits, double* probs) {
  const int C = cfg->channels, L = cfg->num_layers, NH = cfg->num_heads, hs = C / NH;
  const int maxT = cfg->max_seq_len;
  const double scale = 1.0 / sqrt((double)hs);
  OracleParams w = oracle_params(cfg, params);
  double* x = (double*)malloc(sizeof(double) * B * C);
  double* h = (double*)malloc(sizeof(double) * B * C);
  double* qkv = (double*)malloc(sizeof(double) * B * 3 * C);
  double* att = (double*)malloc(sizeof(double) * B * C);
  double* proj = (double*)malloc(sizeof(double) * B * C);
  double* fc = (double*)malloc(sizeof(double) * B * 4 * C);
  double* fcg = (double*)malloc(sizeof(double) * B * 4 * C);
  double* p = (double*)malloc(sizeof(double) * (pos + 1));

  for (int b = 0; b < B; b++)
    for (int c = 0; c < C; c++)
      x[(size_t)b * C + c] = (double)w.wte[(size_t)tok[b] * C + c] + (double)w.wpe[(size_t)pos * C + c];
  for (int l = 0; l < L; l++) {
    oracle_layernorm(h, NULL, NULL, x, w.ln1w + (size_t)l * C, w.ln1b + (size_t)l * C, B, C);
    oracle_matmul(qkv, h, w.qkvw + (size_t)l * 3 * C * C, w.qkvb + (size_t)l * 3 * C, B, C, 3 * C);
    for (int b = 0; b < B; b++)
      for (int hd = 0; hd < NH; hd++) {
        const size_t base = (((size_t)l * B + b) * NH + hd) * maxT;
        for (int d = 0; d < hs; d++) {
          kcache[(base + pos) * hs + d] = qkv[(size_t)b * 3 * C + C + hd * hs + d];
          vcache[(base + pos) * hs + d] = qkv[(size_t)b * 3 * C + 2 * C + hd * hs + d];
        }
        const double* q = qkv + (size_t)b * 3 * C + hd * hs;
        double mx = -INFINITY;
        for (int j = 0; j <= pos; j++) {
          double dot = 0.0;
          for (int d = 0; d < hs; d++) dot += q[d] * kcache[(base + j) * hs + d];
          p[j] = dot * scale;
          if (p[j] > mx) mx = p[j];
        }
        double sum = 0.0;
        for (int j = 0; j <= pos; j++) { p[j] = exp(p[j] - mx); sum += p[j]; }
        for (int d = 0; d < hs; d++) {
          double acc = 0.0;
          for (int j = 0; j <= pos; j++) acc += (p[j] / sum) * vcache[(base + j) * hs + d];
          att[(size_t)b * C + hd * hs + d] = acc;
        }
      }
    oracle_matmul(proj, att, w.attprojw + (size_t)l * C * C, w.attprojb + (size_t)l * C, B, C, C);
    oracle_residual(x, x, proj, B * C);
    oracle_layernorm(h, NULL, NULL, x, w.ln2w + (size_t)l * C, w.ln2b + (size_t)l * C, B, C);
    oracle_matmul(fc, h, w.fcw + (size_t)l * 4 * C * C, w.fcb + (size_t)l * 4 * C, B, C, 4 * C);
    oracle_gelu(fcg, fc, B * 4 * C);
    oracle_matmul(proj, fcg, w.fcprojw + (size_t)l * 4 * C * C, w.fcprojb + (size_t)l * C, B, 4 * C, C);
    oracle_residual(x, x, proj, B * C);
  }
  oracle_layernorm(h, NULL, NULL, x, w.lnfw, w.lnfb, B, C);
  oracle_matmul(logits, h, w.wte, NULL, B, C, cfg->padded_vocab_size);
  if (probs) oracle_softmax(probs, logits, B, cfg->vocab_size, cfg->padded_vocab_size);
  free(x); free(h); free(qkv); free(att); free(proj); free(fc); free(fcg); free(p);
}

/* ====================================================== the training step */
/* The backward pass of the whole model and the optimizer step (llm.c "State
 * of the Union": a GPT-2 training step = forward blocks, the classifier
 * (softmax cross-entropy), backward blocks, AdamW; the per-kernel table
 * names their backward kernels: matmul backward with its bias, layernorm
 * backward, gelu backward, the attention softmax backward, encoder
 * backward).  Each backward below is the chain rule of its forward, written
 * from the forward's definition. */

/* y = x W^T + b:  dx = dy W (set),  dW += dy^T x,  db += sum over rows of dy */
void oracle_matmul_backward(double* dinp, double* dW, double* db, const double* dout, const double* inp,
                            const float* W, int N, int C, int OC) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; n++)
    for (int c = 0; c < C; c++) {
      double acc = 0.0;
      for (int o = 0; o < OC; o++) acc += dout[(size_t)n * OC + o] * (double)W[(size_t)o * C + c];
      dinp[(size_t)n * C + c] = acc;
    }
#pragma omp parallel for schedule(static)
  for (int o = 0; o < OC; o++) {
    for (int c = 0; c < C; c++) {
      double acc = 0.0;
      for (int n = 0; n < N; n++) acc += dout[(size_t)n * OC + o] * inp[(size_t)n * C + c];
      dW[(size_t)o * C + c] += acc;
    }
    if (db) {
      double acc = 0.0;
      for (int n = 0; n < N; n++) acc += dout[(size_t)n * OC + o];
      db[o] += acc;
    }
  }
}

/* y = xhat w + b with xhat = (x - mean) rstd:  dw += sum dy xhat,
 * db += sum dy, and with g = dy w:
 * dx = rstd (g - mean_c(g) - xhat mean_c(g xhat))  (set) */
void oracle_layernorm_backward(double* dinp, double* dw, double* db, const double* dout, const double* inp,
                               const float* w, const double* mean, const double* rstd, int N, int C) {
  for (int n = 0; n < N; n++) {
    const double* x = inp + (size_t)n * C;
    const double* dy = dout + (size_t)n * C;
    double mg = 0.0, mgx = 0.0;
    for (int c = 0; c < C; c++) {
      const double xhat = (x[c] - mean[n]) * rstd[n];
      const double g = dy[c] * (double)w[c];
      mg += g;
      mgx += g * xhat;
      dw[c] += dy[c] * xhat;
      db[c] += dy[c];
    }
    mg /= C;
    mgx /= C;
    for (int c = 0; c < C; c++) {
      const double xhat = (x[c] - mean[n]) * rstd[n];
      dinp[(size_t)n * C + c] = rstd[n] * (dy[c] * (double)w[c] - mg - xhat * mgx);
    }
  }
}

/* d/dx of 0.5 x (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3):
 * 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) sqrt(2/pi) (1 + 3 * 0.044715 x^2) */
void oracle_gelu_backward(double* dinp, const double* inp, const double* dout, int n) {
  const double k = sqrt(2.0 / M_PI);
  for (int i = 0; i < n; i++) {
    const double x = inp[i];
    const double th = tanh(k * (x + 0.044715 * x * x * x));
    const double d = 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * k * (1.0 + 3.0 * 0.044715 * x * x);
    dinp[i] = dout[i] * d;
  }
}

/* One training step's loss and gradient: mean over the B*T positions of the
 * cross-entropy -log probs[n][targets[n]] of the vocabulary softmax, and its
 * gradient with respect to every parameter, in the parameter buffer's
 * layout (grads: double[num_params], overwritten).  The forward keeps every
 * activation the backward needs. */
void oracle_gpt2_forward_backward(const OracleGPT2Config* cfg, const float* params, const int* tok,
                                  const int* targets, int B, int T, double* grads, double* loss_out) {
  const int C = cfg->channels, L = cfg->num_layers, NH = cfg->num_heads;
  const int V = cfg->vocab_size, Vp = cfg->padded_vocab_size;
  const size_t N = (size_t)B * T, NC = N * C;
  OracleParams w = oracle_params(cfg, params);
  /* the gradient buffer, viewed like the parameters */
  const size_t np = oracle_num_params(cfg);
  memset(grads, 0, sizeof(double) * np);
  const size_t o_wte = w.wte - params, o_wpe = w.wpe - params, o_ln1w = w.ln1w - params, o_ln1b = w.ln1b - params,
               o_qkvw = w.qkvw - params, o_qkvb = w.qkvb - params, o_apw = w.attprojw - params,
               o_apb = w.attprojb - params, o_ln2w = w.ln2w - params, o_ln2b = w.ln2b - params,
               o_fcw = w.fcw - params, o_fcb = w.fcb - params, o_fpw = w.fcprojw - params,
               o_fpb = w.fcprojb - params, o_lnfw = w.lnfw - params, o_lnfb = w.lnfb - params;
  /* ---- forward, keeping activations (per layer) */
  double* xin = (double*)malloc(sizeof(double) * (L + 1) * NC);   /* residual stream entering layer l; [L] = final */
  double* xmid = (double*)malloc(sizeof(double) * L * NC);        /* after the attention sub-block */
  double* ln1 = (double*)malloc(sizeof(double) * L * NC);
  double* ln1m = (double*)malloc(sizeof(double) * L * N);
  double* ln1r = (double*)malloc(sizeof(double) * L * N);
  double* qkv = (double*)malloc(sizeof(double) * L * 3 * NC);
  double* att = (double*)malloc(sizeof(double) * L * NC);
  double* ln2 = (double*)malloc(sizeof(double) * L * NC);
  double* ln2m = (double*)malloc(sizeof(double) * L * N);
  double* ln2r = (double*)malloc(sizeof(double) * L * N);
  double* fc = (double*)malloc(sizeof(double) * L * 4 * NC);
  double* fcg = (double*)malloc(sizeof(double) * L * 4 * NC);
  double* lnf = (double*)malloc(sizeof(double) * NC);
  double* lnfm = (double*)malloc(sizeof(double) * N);
  double* lnfr = (double*)malloc(sizeof(double) * N);
  double* logits = (double*)malloc(sizeof(double) * N * Vp);
  double* proj = (double*)malloc(sizeof(double) * NC);
  oracle_encoder(xin, tok, w.wte, w.wpe, B, T, C);
  for (int l = 0; l < L; l++) {
    double* x = xin + (size_t)l * NC;
    double* xm = xmid + (size_t)l * NC;
    oracle_layernorm(ln1 + l * NC, ln1m + l * N, ln1r + l * N, x, w.ln1w + (size_t)l * C, w.ln1b + (size_t)l * C,
                     (int)N, C);
    oracle_matmul(qkv + l * 3 * NC, ln1 + l * NC, w.qkvw + (size_t)l * 3 * C * C, w.qkvb + (size_t)l * 3 * C, (int)N,
                  C, 3 * C);
    oracle_attention(att + l * NC, qkv + l * 3 * NC, B, T, C, NH);
    oracle_matmul(proj, att + l * NC, w.attprojw + (size_t)l * C * C, w.attprojb + (size_t)l * C, (int)N, C, C);
    oracle_residual(xm, x, proj, (int)NC);
    oracle_layernorm(ln2 + l * NC, ln2m + l * N, ln2r + l * N, xm, w.ln2w + (size_t)l * C, w.ln2b + (size_t)l * C,
                     (int)N, C);
    oracle_matmul(fc + l * 4 * NC, ln2 + l * NC, w.fcw + (size_t)l * 4 * C * C, w.fcb + (size_t)l * 4 * C, (int)N, C,
                  4 * C);
    oracle_gelu(fcg + l * 4 * NC, fc + l * 4 * NC, (int)(4 * NC));
    oracle_matmul(proj, fcg + l * 4 * NC, w.fcprojw + (size_t)l * 4 * C * C, w.fcprojb + (size_t)l * C, (int)N,
                  4 * C, C);
    oracle_residual(xin + (size_t)(l + 1) * NC, xm, proj, (int)NC);
  }
  oracle_layernorm(lnf, lnfm, lnfr, xin + (size_t)L * NC, w.lnfw, w.lnfb, (int)N, C);
  oracle_matmul(logits, lnf, w.wte, NULL, (int)N, C, Vp);
  /* ---- the loss and dL/dlogits (softmax cross-entropy, mean over rows) */
  double loss = 0.0;
  for (size_t n = 0; n < N; n++) {
    double* lg = logits + n * Vp;
    double mx = -INFINITY;
    for (int v = 0; v < V; v++) if (lg[v] > mx) mx = lg[v];
    double sum = 0.0;
    for (int v = 0; v < V; v++) sum += exp(lg[v] - mx);
    loss += -(lg[targets[n]] - mx - log(sum));
    for (int v = 0; v < Vp; v++) {  /* logits become dlogits */
      const double p = v < V ? exp(lg[v] - mx) / sum : 0.0;
      lg[v] = (p - (v == targets[n] ? 1.0 : 0.0)) / (double)N;
    }
  }
  *loss_out = loss / (double)N;
  /* ---- backward */
  double* dx = (double*)malloc(sizeof(double) * NC);
  double* dh = (double*)malloc(sizeof(double) * NC);
  double* dt = (double*)malloc(sizeof(double) * 4 * NC);
  double* dt2 = (double*)malloc(sizeof(double) * 4 * NC);
  double* dqkv = (double*)malloc(sizeof(double) * 3 * NC);
  /* the tied LM head: logits = lnf wte^T */
  oracle_matmul_backward(dh, grads + o_wte, NULL, logits, lnf, w.wte, (int)N, C, Vp);
  oracle_layernorm_backward(dx, grads + o_lnfw, grads + o_lnfb, dh, xin + (size_t)L * NC, w.lnfw, lnfm, lnfr, (int)N,
                            C);
  for (int l = L - 1; l >= 0; l--) {
    /* x_out = x_mid + fcproj(GELU(fc(LN2(x_mid)))): dx is dL/dx_out */
    oracle_matmul_backward(dt, grads + o_fpw + (size_t)l * 4 * C * C, grads + o_fpb + (size_t)l * C, dx,
                           fcg + l * 4 * NC, w.fcprojw + (size_t)l * 4 * C * C, (int)N, 4 * C, C);
    oracle_gelu_backward(dt2, fc + l * 4 * NC, dt, (int)(4 * NC));
    oracle_matmul_backward(dh, grads + o_fcw + (size_t)l * 4 * C * C, grads + o_fcb + (size_t)l * 4 * C, dt2,
                           ln2 + l * NC, w.fcw + (size_t)l * 4 * C * C, (int)N, C, 4 * C);
    oracle_layernorm_backward(dt, grads + o_ln2w + (size_t)l * C, grads + o_ln2b + (size_t)l * C, dh,
                              xmid + (size_t)l * NC, w.ln2w + (size_t)l * C, ln2m + l * N, ln2r + l * N, (int)N, C);
    for (size_t i = 0; i < NC; i++) dx[i] += dt[i];  /* dL/dx_mid: the residual path plus the MLP's */
    /* x_mid = x_in + attproj(attention(qkv(LN1(x_in)))) */
    oracle_matmul_backward(dh, grads + o_apw + (size_t)l * C * C, grads + o_apb + (size_t)l * C, dx, att + l * NC,
                           w.attprojw + (size_t)l * C * C, (int)N, C, C);
    oracle_attention_backward(dqkv, dh, qkv + l * 3 * NC, B, T, C, NH);
    oracle_matmul_backward(dh, grads + o_qkvw + (size_t)l * 3 * C * C, grads + o_qkvb + (size_t)l * 3 * C, dqkv,
                           ln1 + l * NC, w.qkvw + (size_t)l * 3 * C * C, (int)N, C, 3 * C);
    oracle_layernorm_backward(dt, grads + o_ln1w + (size_t)l * C, grads + o_ln1b + (size_t)l * C, dh,
                              xin + (size_t)l * NC, w.ln1w + (size_t)l * C, ln1m + l * N, ln1r + l * N, (int)N, C);
    for (size_t i = 0; i < NC; i++) dx[i] += dt[i];  /* dL/dx_in */
  }
  /* the encoder: x = wte[tok] + wpe[t] */
  for (int b = 0; b < B; b++)
    for (int t = 0; t < T; t++) {
      const size_t n = (size_t)b * T + t;
      for (int c = 0; c < C; c++) {
        grads[o_wte + (size_t)tok[n] * C + c] += dx[n * C + c];
        grads[o_wpe + (size_t)t * C + c] += dx[n * C + c];
      }
    }
  free(xin); free(xmid); free(ln1); free(ln1m); free(ln1r); free(qkv); free(att); free(ln2); free(ln2m);
  free(ln2r); free(fc); free(fcg); free(lnf); free(lnfm); free(lnfr); free(logits); free(proj);
  free(dx); free(dh); free(dt); free(dt2); free(dqkv);
}

/* AdamW (Loshchilov and Hutter, "Decoupled Weight Decay Regularization",
 * Algorithm 2), step t >= 1, the same decay for every parameter:
 *   m = b1 m + (1 - b1) g,  v = b2 v + (1 - b2) g^2,
 *   mhat = m / (1 - b1^t),  vhat = v / (1 - b2^t),
 *   p -= lr (mhat / (sqrt(vhat) + eps) + wd p). */
void oracle_adamw(double* p, const double* g, double* m, double* v, size_t n, double lr, double b1, double b2,
                  double eps, double wd, int t) {
  const double c1 = 1.0 - pow(b1, t), c2 = 1.0 - pow(b2, t);
  for (size_t i = 0; i < n; i++) {
    m[i] = b1 * m[i] + (1.0 - b1) * g[i];
    v[i] = b2 * v[i] + (1.0 - b2) * g[i] * g[i];
    p[i] -= lr * ((m[i] / c1) / (sqrt(v[i] / c2) + eps) + wd * p[i]);
  }
}
