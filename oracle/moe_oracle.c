/*
 * moe_oracle.c — float64 CPU oracle of one mixture-of-experts layer over a
 * verification pass.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only tests/, the smoke check in __graft_entry__ and the CPU
 * baseline leg of bench.py do. It shares no code, header, table or helper
 * with the CUDA library: it is the plain definition written out with straight
 * loops in double precision, so that a reader can check it against the
 * sources by eye.
 *
 * Sources (page title, then section):
 *   [G] "Deep Dive into Mixture of Experts: From 1991 to DeepSeek-V3",
 *       §2 "The Sparse-Gating Leap", top-k gating sketch: logits = x·W_g,
 *       keep the top k, softmax over just the k kept logits, output =
 *       Σ weight·expert(x).
 *   [S] same post, §5 "DeepSeek-V3 and the Current State of the Art", routing
 *       sketch: output starts from the sum of the always-on shared experts.
 *   [G'] same post, §5, routing sketch: a per-expert bias added to the gate's
 *       scores before the top-k; the sketch takes the softmax over the kept
 *       biased scores.
 *   [D] same post, §1 "1991: Where It Started": the dense mixture, where every
 *       expert runs and the gate weights combine them.
 *   [B] "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes,
 *       Kernel Bandwidth and the Best Draft Length", abstract: per-slot bytes
 *       (an expert read once per token) and dedup bytes (each selected expert
 *       read once per pass).
 * Readings where the sources are silent:
 *   - experts are SwiGLU FFNs without biases: W_down(silu(W_gate x) ⊙ W_up x),
 *     silu(z) = z/(1+exp(-z)); the sources never define the expert body.
 *   - equal logits are ordered by ascending expert index (ties select the
 *     lower index).
 *   - shared experts carry weight 1 (the [S] sketch adds s(x) unweighted).
 *
 * Parity pins: every function here is checked in tests/test_oracle.py
 * against something other than itself (brute force over subsets, torch's
 * float64 linear/silu/softmax/topk, the dense formulation of [D], Python
 * sets, closed forms). No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Weight element i of a row-major matrix stored as fp32 (wdtype 0) or as
 * bfloat16 bit patterns (wdtype 1). bfloat16 -> double is exact: the 16 bits
 * are the top half of an IEEE binary32. */
static double weight_at(const void* w, int wdtype, size_t i) {
  if (wdtype == 0) return (double)((const float*)w)[i];
  uint32_t bits = ((uint32_t)((const uint16_t*)w)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* [G] logits = x·W_g:  logits[t][e] = Σ_i x[t][i]·W_g[e][i], in double.
 * Also writes absdot[t][e] = Σ_i |x[t][i]·W_g[e][i]| when absdot != NULL,
 * which bounds the rounding error of any fp32 evaluation of the same dot. */
int oracle_gate_logits(int d, int E, int n, const float* x, const float* wg, double* logits,
                       double* absdot) {
  if (d <= 0 || E <= 0 || n <= 0 || !x || !wg || !logits) return 1;
  for (int t = 0; t < n; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0, a = 0.0;
      for (int i = 0; i < d; ++i) {
        double p = (double)x[(size_t)t * d + i] * (double)wg[(size_t)e * d + i];
        s += p;
        a += fabs(p);
      }
      logits[(size_t)t * E + e] = s;
      if (absdot) absdot[(size_t)t * E + e] = a;
    }
  }
  return 0;
}

/* Order used by the selection: larger logit first; equal logits by the lower
 * expert index. qsort over (logit, index) records. */
typedef struct {
  double v;
  int e;
} scored;

static int by_logit_then_index(const void* pa, const void* pb) {
  const scored* a = (const scored*)pa;
  const scored* b = (const scored*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->e < b->e) ? -1 : (a->e > b->e);
}

/* [G] top_k_vals, top_k_idx = topk(logits, k); top_k_weights =
 * softmax(top_k_vals), i.e. a softmax over the k kept logits only.
 *   idx[t][j]  j-th selected expert (descending logit, ties -> lower index)
 *   w[t][j]    exp(l_j - l_max) / Σ_{j'<k} exp(l_j' - l_max)
 *   gap[t]     (may be NULL) smallest difference between consecutive logits
 *              in the sorted order among positions 0..k (position k is the
 *              first expert left out; +inf when k == E and k == 1). A GPU
 *              evaluation whose logit error is below gap/2 orders these
 *              positions exactly as this function does.                    */
int oracle_topk_biased(int E, int k, int n, const double* logits, const double* bias,
                       int bias_in_weights, int32_t* idx, double* w, double* gap);

int oracle_topk(int E, int k, int n, const double* logits, int32_t* idx, double* w, double* gap) {
  return oracle_topk_biased(E, k, n, logits, NULL, 1, idx, w, gap);
}

/* [G'] the DeepSeek-style routing sketch: a per-expert bias b_e is added to
 * the gate's scores and the top k of l_e + b_e are selected (ties -> lower
 * index). bias_in_weights = 1 takes the softmax over the k kept biased
 * scores, as the sketch writes it; 0 takes it over the kept experts'
 * unbiased logits (bias for selection only). bias == NULL is no bias. gap is
 * that of the biased scores (the values the selection compares).          */
int oracle_topk_biased(int E, int k, int n, const double* logits, const double* bias,
                       int bias_in_weights, int32_t* idx, double* w, double* gap) {
  if (E <= 0 || k <= 0 || k > E || n <= 0 || !logits || !idx || !w) return 1;
  scored* s = (scored*)malloc(sizeof(scored) * (size_t)E);
  double* u = (double*)malloc(sizeof(double) * (size_t)k);
  if (!s || !u) {
    free(s);
    free(u);
    return 2;
  }
  for (int t = 0; t < n; ++t) {
    for (int e = 0; e < E; ++e) {
      s[e].v = logits[(size_t)t * E + e] + (bias ? bias[e] : 0.0);
      s[e].e = e;
    }
    qsort(s, (size_t)E, sizeof(scored), by_logit_then_index);
    /* the values the softmax runs over, and their maximum */
    double umax = -INFINITY, z = 0.0;
    for (int j = 0; j < k; ++j) {
      u[j] = (bias && !bias_in_weights) ? logits[(size_t)t * E + s[j].e] : s[j].v;
      if (u[j] > umax) umax = u[j];
    }
    for (int j = 0; j < k; ++j) z += exp(u[j] - umax);
    for (int j = 0; j < k; ++j) {
      idx[(size_t)t * k + j] = s[j].e;
      w[(size_t)t * k + j] = exp(u[j] - umax) / z;
    }
    if (gap) {
      int last = (k < E) ? k : E - 1;
      double g = INFINITY;
      for (int j = 0; j < last; ++j) {
        double dj = s[j].v - s[j + 1].v;
        if (dj < g) g = dj;
      }
      gap[t] = g;
    }
  }
  free(s);
  free(u);
  return 0;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* One expert on one hidden state (the SwiGLU reading above):
 *   g_i = Σ_c W_gate[i][c]·x_c,  u_i = Σ_c W_up[i][c]·x_c   (i < I, c < d)
 *   h_i = silu(g_i)·u_i
 *   out_r = Σ_i W_down[r][i]·h_i                            (r < d)
 * wgate, wup: [I][d]; wdown: [d][I]; elements in wdtype.                  */
int oracle_expert_ffn(int d, int I, int wdtype, const void* wgate, const void* wup,
                      const void* wdown, const double* x, double* out) {
  if (d <= 0 || I <= 0 || !wgate || !wup || !wdown || !x || !out) return 1;
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  if (!h) return 2;
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < d; ++c) {
      g += weight_at(wgate, wdtype, (size_t)i * d + c) * x[c];
      u += weight_at(wup, wdtype, (size_t)i * d + c) * x[c];
    }
    h[i] = silu(g) * u;
  }
  for (int r = 0; r < d; ++r) {
    double o = 0.0;
    for (int i = 0; i < I; ++i) o += weight_at(wdown, wdtype, (size_t)r * I + i) * h[i];
    out[r] = o;
  }
  free(h);
  return 0;
}

/* [G]+[S] output of the layer for one token given its selection:
 *   y = Σ_{i<s} FFN_shared_i(x) + Σ_{j<k} w_j·FFN_{idx_j}(x)
 * Expert e's matrices start at element e·I·d of wgate/wup/wdown ([E][I][d],
 * [E][I][d], [E][d][I]); shared expert i's at i·I·d of wsg/wsu/wsd.
 * slot_out (may be NULL) receives [k+s][d]: slot j < k = w_j·FFN_{idx_j}(x),
 * slot k+i = FFN_shared_i(x).                                              */
int oracle_moe_token(int d, int I, int k, int s, int wdtype, const void* wgate, const void* wup,
                     const void* wdown, const void* wsg, const void* wsu, const void* wsd,
                     const float* x_t, const int32_t* idx_t, const double* w_t, double* y,
                     double* slot_out) {
  if (d <= 0 || I <= 0 || k <= 0 || s < 0 || !x_t || !idx_t || !w_t || !y) return 1;
  size_t esz = (size_t)I * d * (wdtype == 0 ? 4 : 2); /* bytes of one matrix of one expert */
  double* xd = (double*)malloc(sizeof(double) * (size_t)d);
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  if (!xd || !o) {
    free(xd);
    free(o);
    return 2;
  }
  for (int c = 0; c < d; ++c) xd[c] = (double)x_t[c];
  for (int r = 0; r < d; ++r) y[r] = 0.0;
  for (int i = 0; i < s; ++i) {
    oracle_expert_ffn(d, I, wdtype, (const char*)wsg + i * esz, (const char*)wsu + i * esz,
                      (const char*)wsd + i * esz, xd, o);
    for (int r = 0; r < d; ++r) {
      y[r] += o[r];
      if (slot_out) slot_out[(size_t)(k + i) * d + r] = o[r];
    }
  }
  for (int j = 0; j < k; ++j) {
    int e = idx_t[j];
    oracle_expert_ffn(d, I, wdtype, (const char*)wgate + e * esz, (const char*)wup + e * esz,
                      (const char*)wdown + e * esz, xd, o);
    for (int r = 0; r < d; ++r) {
      y[r] += w_t[j] * o[r];
      if (slot_out) slot_out[(size_t)j * d + r] = w_t[j] * o[r];
    }
  }
  free(xd);
  free(o);
  return 0;
}

/* [D] dense mixture for one token: every expert runs and is weighted by
 * gate[e] (gate[e] = 0 for experts the sparse gate did not select). Shared
 * experts are added as in oracle_moe_token. Used only to pin the sparse form. */
int oracle_dense_token(int d, int I, int E, int s, int wdtype, const void* wgate, const void* wup,
                       const void* wdown, const void* wsg, const void* wsu, const void* wsd,
                       const float* x_t, const double* gate, double* y) {
  if (d <= 0 || I <= 0 || E <= 0 || s < 0 || !x_t || !gate || !y) return 1;
  size_t esz = (size_t)I * d * (wdtype == 0 ? 4 : 2);
  double* xd = (double*)malloc(sizeof(double) * (size_t)d);
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  if (!xd || !o) {
    free(xd);
    free(o);
    return 2;
  }
  for (int c = 0; c < d; ++c) xd[c] = (double)x_t[c];
  for (int r = 0; r < d; ++r) y[r] = 0.0;
  for (int i = 0; i < s; ++i) {
    oracle_expert_ffn(d, I, wdtype, (const char*)wsg + i * esz, (const char*)wsu + i * esz,
                      (const char*)wsd + i * esz, xd, o);
    for (int r = 0; r < d; ++r) y[r] += o[r];
  }
  for (int e = 0; e < E; ++e) {
    oracle_expert_ffn(d, I, wdtype, (const char*)wgate + e * esz, (const char*)wup + e * esz,
                      (const char*)wdown + e * esz, xd, o);
    for (int r = 0; r < d; ++r) y[r] += gate[e] * o[r];
  }
  free(xd);
  free(o);
  return 0;
}

/* [B] union of the experts selected in one pass, and the (token, slot) pairs
 * grouped by expert.
 *   union_ids[0..*count)   the distinct values of idx, ascending
 *   offsets[0..*count]     pairs of union_ids[u] occupy rows offsets[u]..offsets[u+1]-1
 *   pair_tok/pair_slot     those pairs, ordered by (expert, token)
 * Counting sort by expert over the pairs taken in token-major order.       */
int oracle_union(int E, int k, int n, const int32_t* idx, int32_t* union_ids, int32_t* count,
                 int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot) {
  if (E <= 0 || k <= 0 || n <= 0 || !idx || !union_ids || !count || !offsets || !pair_tok ||
      !pair_slot)
    return 1;
  int* per_expert = (int*)calloc((size_t)E, sizeof(int));
  if (!per_expert) return 2;
  for (int p = 0; p < n * k; ++p) {
    if (idx[p] < 0 || idx[p] >= E) {
      free(per_expert);
      return 3;
    }
    per_expert[idx[p]] += 1;
  }
  int u = 0, row = 0;
  for (int e = 0; e < E; ++e) {
    if (per_expert[e] == 0) continue;
    union_ids[u] = e;
    offsets[u] = row;
    for (int t = 0; t < n; ++t)
      for (int j = 0; j < k; ++j)
        if (idx[(size_t)t * k + j] == e) {
          pair_tok[row] = t;
          pair_slot[row] = j;
          ++row;
        }
    ++u;
  }
  offsets[u] = row;
  *count = u;
  free(per_expert);
  return 0;
}

/* [B] expert-weight bytes requested in one pass:
 *   bytes[0] per-slot = n·k·E_b   (each slot reads its expert)
 *   bytes[1] dedup    = |U|·E_b   (each distinct expert read once)
 *   bytes[2] shared   = s·E_b     (read once per pass by either engine)
 * with E_b = 3·d·I·(bytes per weight). */
int oracle_bytes(int d, int I, int k, int s, int n, int wdtype, int union_count,
                 uint64_t* bytes) {
  if (!bytes) return 1;
  uint64_t eb = 3ull * (uint64_t)d * (uint64_t)I * (wdtype == 0 ? 4ull : 2ull);
  bytes[0] = (uint64_t)n * (uint64_t)k * eb;
  bytes[1] = (uint64_t)union_count * eb;
  bytes[2] = (uint64_t)s * eb;
  return 0;
}
