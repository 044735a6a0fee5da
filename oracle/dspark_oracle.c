/*
 * dspark_oracle.c -- CPU oracle for DSpark ancestral draft-block sampling.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference legs use it.  It shares no code, header, table or
 * constant generator with the CUDA path under ancestral_draft_sampling_gb300/.
 *
 * A plain, slow, obviously-correct restatement of what the method computes,
 * in the order the pages state it:
 *
 *   brb-nv/TensorRT-LLM PR #21, "2. Golden sampling semantics":
 *     position k is drawn from softmax((base_k + bias(d_{k-1})) / T), where
 *     d_{k-1} is the token drawn just before it; drafts use the temperature
 *     only (no top-k / top-p / min-p); greedy requests draft the argmax chain;
 *     the distribution each draft was drawn from is stored as its proposal.
 *   brb-nv/TensorRT-LLM PR #27, "2. One fused kernel per draft position":
 *     add the Markov bias, scale by 1/T, take the argmax of the scaled logits
 *     plus Gumbel noise from a counter-based Philox stream keyed by the
 *     request's (seed, offset) draft slot of position k; biased logits are
 *     kept in float32; afterwards q_k = softmax(logits_k / T) is written from
 *     those float32 logits, recomputing logits_k / T bit for bit; CUDA-graph
 *     padding rows draw from the bias alone.  Results table: the Markov head
 *     is rank 256 ("rank-256 Markov head").
 *   brb-nv/TensorRT-LLM PR #21, "2. Golden sampling semantics": the default
 *     verification rule is standard token-level rejection sampling; the
 *     block rule is the block verification of Sun et al. (2024).
 *
 * Readings where the pages are silent:
 *   - Philox variant: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 *     random numbers: as easy as 1, 2, 3", SC'11).
 *   - Counter layout: key = (seed lo, seed hi); counter =
 *     (v >> 2, k | stream << 16, offset lo, offset hi), word v & 3.
 *     stream 0 = draft noise, 1 = acceptance uniforms, 2 = residual / bonus
 *     noise.
 *   - Gumbel transform: w = (x + 0.5) * 2^-32, g = -log(-log1p(-w)).
 *   - The scaled logit is the float32 IEEE quotient l / T (pages: "bit for
 *     bit").  The perturbed score that decides the token is taken in the
 *     kernel's precision: g is computed in double and rounded once to float,
 *     and score = s + g is a float32 addition.  Ties go to the lowest index;
 *     a NaN or -inf score never wins, and a row where nothing wins draws
 *     token 0.
 *   - Greedy rows consume no noise and store a one-hot proposal (PR #27,
 *     "Also checked": a greedy-sentinel row draws the argmax with a one-hot
 *     proposal).
 *   - Padding rows ignore the drafter logits (even NaN) and use l = bias.
 *   - Bias: accumulated in double over j = 0..r-1, then l = base + bias is
 *     rounded once to float.
 *   - Verification uniforms: u = ((x >> 9) + 0.5) * 2^-23, exact in float;
 *     accept iff float(u * q[d]) < p[d].
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off (no -ffast-math: IEEE float
 * division and the libm log/exp are relied on).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* ---------------------------------------------------------------- Philox */

/* Philox4x32-10, SC'11 paper: the round multipliers and the Weyl key
 * increments are the published constants of the Philox-4x32 family. */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { /* the key is bumped between rounds */
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The raw 32-bit word that feeds element `index` of stream `stream` at
 * position k of request (seed, offset). */
uint32_t oracle_noise_word(uint64_t seed, uint64_t offset, int k, int stream,
                           uint32_t index) {
  uint32_t ctr[4], key[2], out[4];
  ctr[0] = index >> 2;
  ctr[1] = (uint32_t)k | ((uint32_t)stream << 16);
  ctr[2] = (uint32_t)(offset & 0xffffffffu);
  ctr[3] = (uint32_t)(offset >> 32);
  key[0] = (uint32_t)(seed & 0xffffffffu);
  key[1] = (uint32_t)(seed >> 32);
  oracle_philox4x32_10(ctr, key, out);
  return out[index & 3u];
}

/* The words of elements 0 .. n-1 (oracle_noise_word for each index), for
 * comparisons over long stretches of counters. */
void oracle_noise_words(uint64_t seed, uint64_t offset, int k, int stream,
                        uint32_t n, uint32_t* out) {
  for (uint32_t i = 0; i < n; ++i)
    out[i] = oracle_noise_word(seed, offset, k, stream, i);
}

/* Standard Gumbel variate from one 32-bit word: w uniform in (0, 1),
 * g = -log(-log(1 - w)). */
double oracle_gumbel(uint32_t x) {
  double w = ((double)x + 0.5) * 0x1p-32;
  double e = -log1p(-w);
  return -log(e);
}

/* Uniform in (0, 1) for the acceptance test; exact in float and double. */
float oracle_accept_uniform(uint32_t x) {
  return (float)(((double)(x >> 9) + 0.5) * 0x1p-23);
}

/* ------------------------------------------------------------- helpers */

static double load_elem(const void* p, int dtype, size_t i) {
  if (dtype == ORACLE_F32) return (double)((const float*)p)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------- one draft position */

/* The decision and the proposal of one row from its float32 logits: the
 * argmax of s = l / T (greedy) or of float(s + g) with g the Gumbel variate
 * of noise `stream` at position k (sampled), lowest index on ties, NaN and
 * -inf never winning; and q = softmax(s) in double (one-hot for greedy).
 * Shared by the draft positions (stream 0) and the temperature-only target
 * sampler (stream 3). */
static void oracle_sample_row(const float* logits, int V, uint64_t seed,
                              uint64_t offset, int k, int stream, float T,
                              int greedy, double* probs_out, int* token_out,
                              double* M_out, double* S_out, float* best_out,
                              float* second_out) {
  /* decision: argmax of s (greedy) or of float(s + g) (sampled) */
  int token = 0;
  float best = -INFINITY;
  int found = 0;
  for (int v = 0; v < V; ++v) {
    float s = logits[v] / T;
    float score;
    if (greedy) {
      score = s;
    } else {
      float g = (float)oracle_gumbel(oracle_noise_word(seed, offset, k, stream,
                                                       (uint32_t)v));
      score = s + g;
    }
    if (score > best) { /* NaN and -inf never win; ties keep the lower v */
      best = score;
      token = v;
      found = 1;
    }
  }
  float second = -INFINITY;
  for (int v = 0; v < V; ++v) {
    if (v == token) continue;
    float s = logits[v] / T;
    float score = s;
    if (!greedy)
      score = s + (float)oracle_gumbel(
                      oracle_noise_word(seed, offset, k, stream, (uint32_t)v));
    if (!isnan(score) && score > second) second = score;
  }

  /* proposal q = softmax(s) in double from the float32 s */
  double M = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double s = (double)(logits[v] / T);
    if (!isnan(s) && s > M) M = s;
  }
  double S = 0.0;
  for (int v = 0; v < V; ++v) S += exp((double)(logits[v] / T) - M);
  if (greedy) {
    for (int v = 0; v < V; ++v) probs_out[v] = (v == token) ? 1.0 : 0.0;
  } else {
    for (int v = 0; v < V; ++v)
      probs_out[v] = exp((double)(logits[v] / T) - M) / S;
  }

  *token_out = token;
  *M_out = M;
  *S_out = S;
  *best_out = found ? best : -INFINITY;
  *second_out = second;
}

/*
 * One draft position of one request.
 *
 * base_row : [V] drafter logits of this (request, position), dtype base_dtype;
 *            ignored when is_pad != 0 (may be NULL then).
 * U        : [V, r] row-major, Wb : [r, V] row-major, both of dtype w_dtype.
 * prev     : the token drawn just before this position (d0 for position 0).
 * Outputs  : logits_out [V] float32 biased logits l,
 *            probs_out [V] proposal q in double (one-hot for greedy rows),
 *            *token_out, *M_out = max s, *S_out = sum exp(s - M),
 *            *best_out / *second_out = the two largest decision scores
 *            (float32 s + g for sampled rows, s for greedy rows; second is
 *            the largest over v != token, -inf when V == 1).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_draft_position(const void* base_row, int base_dtype, int is_pad,
                          const void* U, const void* Wb, int w_dtype, int V,
                          int r, int prev, uint64_t seed, uint64_t offset,
                          int k, float T, int greedy, float* logits_out,
                          double* probs_out, int* token_out, double* M_out,
                          double* S_out, float* best_out, float* second_out,
                          double* bias_scratch /* [V] */) {
  if (V <= 0 || r <= 0 || prev < 0 || prev >= V || !(T > 0.0f) ||
      !isfinite(T) || U == NULL || Wb == NULL || bias_scratch == NULL ||
      (!is_pad && base_row == NULL))
    return -1;

  /* bias(d) = U[d] @ Wb, accumulated in double in the order j = 0..r-1 */
  for (int v = 0; v < V; ++v) bias_scratch[v] = 0.0;
  for (int j = 0; j < r; ++j) {
    double u = load_elem(U, w_dtype, (size_t)prev * (size_t)r + (size_t)j);
    for (int v = 0; v < V; ++v)
      bias_scratch[v] += u * load_elem(Wb, w_dtype, (size_t)j * (size_t)V + v);
  }

  /* l = base + bias, rounded once to float; padding rows use the bias alone */
  for (int v = 0; v < V; ++v) {
    double base = is_pad ? 0.0 : load_elem(base_row, base_dtype, (size_t)v);
    logits_out[v] = (float)(base + bias_scratch[v]);
  }

  oracle_sample_row(logits_out, V, seed, offset, k, 0, T, greedy, probs_out,
                    token_out, M_out, S_out, best_out, second_out);
  return 0;
}

/* ------------------------------------------------------- whole draft block */

/*
 * The ancestral draft block: for every request b, positions k = 0..K-1 in
 * order, each conditioned on the token drawn before it (d0[b] for k = 0).
 *
 * base [B,K,V] (base_dtype), U [V,r], Wb [r,V] (w_dtype), d0/seed/offset [B],
 * greedy/pad_row [B] or NULL.  Outputs: tokens [B,K], logits [B,K,V] float32, probs [B,K,V] double,
 * rowstats [B,K,2] (M, S) double, top2 [B,K,2] float (best, second) or NULL.
 */
int oracle_draft_block(const void* base, int base_dtype, const void* U,
                       const void* Wb, int w_dtype, const int32_t* d0,
                       const uint64_t* seed, const uint64_t* offset, float T,
                       const uint8_t* greedy, const uint8_t* pad_row, int B,
                       int K, int V, int r, int32_t* tokens, float* logits, double* probs,
                       double* rowstats, float* top2, double* bias_scratch) {
  if (B <= 0 || K <= 0) return -1;
  size_t elt = (base_dtype == ORACLE_F32) ? 4 : 2;
  for (int b = 0; b < B; ++b) {
    int prev = d0[b];
    int is_pad = pad_row ? pad_row[b] != 0 : 0;
    int is_greedy = greedy ? greedy[b] != 0 : 0;
    for (int k = 0; k < K; ++k) {
      size_t row = (size_t)b * (size_t)K + (size_t)k;
      const void* base_row =
          is_pad ? NULL : (const char*)base + row * (size_t)V * elt;
      int token;
      double M, S;
      float best, second;
      int rc = oracle_draft_position(
          base_row, base_dtype, is_pad, U, Wb, w_dtype, V, r, prev, seed[b],
          offset[b], k, T, is_greedy, logits + row * (size_t)V,
          probs + row * (size_t)V, &token, &M, &S, &best, &second,
          bias_scratch);
      if (rc) return rc;
      tokens[row] = token;
      if (rowstats) {
        rowstats[2 * row] = M;
        rowstats[2 * row + 1] = S;
      }
      if (top2) {
        top2[2 * row] = best;
        top2[2 * row + 1] = second;
      }
      prev = token;
    }
  }
  return 0;
}

/* -------------------------------------------------- standard verification */

/* Gumbel-max draw from the unnormalised weights w[0..V-1] >= 0 with stream 2
 * noise at position kk: argmax of float(log w) + float(g), lowest index on
 * ties, zero weights never win.  Returns -1 when every weight is zero. */
static int gumbel_max_weights(const float* w, int V, uint64_t seed,
                              uint64_t offset, int kk, float* best_out,
                              float* second_out) {
  int token = -1;
  float best = -INFINITY, second = -INFINITY;
  for (int v = 0; v < V; ++v) {
    if (!(w[v] > 0.0f)) continue;
    float lw = (float)log((double)w[v]);
    float g = (float)oracle_gumbel(
        oracle_noise_word(seed, offset, kk, 2, (uint32_t)v));
    float score = lw + g;
    if (token < 0 || score > best) {
      if (token >= 0) second = best;
      best = score;
      token = v;
    } else if (score > second) {
      second = score;
    }
  }
  if (best_out) *best_out = best;
  if (second_out) *second_out = second;
  return token;
}

/*
 * Standard token-level rejection sampling (the default "standard" rule of
 * PR #21, "2. Golden sampling semantics"; Leviathan et al. 2023, Chen et al.
 * 2023).  For k = 0..K-1: draft d = tokens[b,k] is accepted iff
 * float(u_k * q_k[d]) < p_k[d] with u_k uniform (stream 1, word 0).  At the
 * first rejection the emitted token is drawn from norm(max(p_k - q_k, 0))
 * (from p_k if that residual is all zero) and accepted_len = k; if all K are
 * accepted the emitted token is drawn from the bonus row p_K and
 * accepted_len = K.  Draws use Gumbel-max with stream 2 noise at position k
 * (K for the bonus row).
 *
 * draft_probs [B,K,V], target_probs [B,K+1,V] float32, tokens [B,K].
 * emit_top2 [B,2] or NULL receives the two largest scores of the emitting
 * draw.  Returns 0, or -1 on a bad argument.
 */
int oracle_verify_standard(const float* draft_probs, const float* target_probs,
                           const int32_t* tokens, const uint64_t* seed,
                           const uint64_t* offset, int B, int K, int V,
                           int32_t* accepted_len, int32_t* emitted,
                           float* emit_top2, float* residual_scratch) {
  if (B <= 0 || K <= 0 || V <= 0) return -1;
  for (int b = 0; b < B; ++b) {
    int acc = K;
    int emit = -1;
    float best = -INFINITY, second = -INFINITY;
    for (int k = 0; k < K; ++k) {
      int d = tokens[(size_t)b * K + k];
      if (d < 0 || d >= V) return -1;
      const float* q = draft_probs + ((size_t)b * K + k) * (size_t)V;
      const float* p = target_probs + ((size_t)b * (K + 1) + k) * (size_t)V;
      float u = oracle_accept_uniform(
          oracle_noise_word(seed[b], offset[b], k, 1, 0u));
      float uq = u * q[d];
      if (uq < p[d]) continue; /* accepted */
      acc = k;
      int any = 0;
      for (int v = 0; v < V; ++v) {
        float diff = p[v] - q[v];
        residual_scratch[v] = diff > 0.0f ? diff : 0.0f;
        if (residual_scratch[v] > 0.0f) any = 1;
      }
      const float* w = any ? residual_scratch : p;
      emit = gumbel_max_weights(w, V, seed[b], offset[b], k, &best, &second);
      break;
    }
    if (acc == K) {
      const float* pK = target_probs + ((size_t)b * (K + 1) + K) * (size_t)V;
      emit = gumbel_max_weights(pK, V, seed[b], offset[b], K, &best, &second);
    }
    accepted_len[b] = acc;
    emitted[b] = emit < 0 ? 0 : emit;
    if (emit_top2) {
      emit_top2[2 * b] = best;
      emit_top2[2 * b + 1] = second;
    }
  }
  return 0;
}

/* ----------------------------------------------------- block verification */

/*
 * Block verification: the block value of rejection_sample_method in PR #21,
 * "2. Golden sampling semantics", which the pages identify as the block
 * verification of Sun et al. (2024) and test for losslessness by chi-square
 * (Test Coverage).  The pages name the rule only; this is the published
 * algorithm restated, with
 * 0-based positions (q_k = draft_probs[b,k], p_k = target_probs[b,k],
 * d_k = tokens[b,k]):
 *
 *   w_0 = 1;  w_{k+1} = min(w_k * (p_k[d_k] / q_k[d_k]), 1)   (k = 0..K-1)
 *   for i = 1..K-1:  r_i = sum_x max(w_i p_i(x) - q_i(x), 0)
 *                    h_i = r_i / (r_i + 1 - w_i)   (1 when r_i = 1 - w_i = 0)
 *   h_K = w_K
 *   accepted_len tau = the largest i in 1..K with eta_i <= h_i (0 if none),
 *   eta_i the stream-1 uniform of position i-1 (the standard rule's u_{i-1});
 *   emitted: drawn from p_K when tau = K, else from norm(max(w_tau p_tau -
 *   q_tau, 0)) (from p_tau if that is all zero), by Gumbel-max with stream-2
 *   noise at position tau.
 *
 * Arithmetic: the w chain and every per-entry term in float32 (a quotient,
 * a product, a difference, each rounded once; a NaN w or term counts as 0);
 * the sums r_i and h_i in double.  h_out [B,K] (or NULL) receives h_1..h_K,
 * eta_out [B,K] (or NULL) eta_1..eta_K.  Returns 0, or -1 on a bad argument.
 */
int oracle_verify_block(const float* draft_probs, const float* target_probs,
                        const int32_t* tokens, const uint64_t* seed,
                        const uint64_t* offset, int B, int K, int V,
                        int32_t* accepted_len, int32_t* emitted,
                        float* emit_top2, double* h_out, float* eta_out,
                        float* residual_scratch) {
  if (B <= 0 || K <= 0 || V <= 0) return -1;
  for (int b = 0; b < B; ++b) {
    const float* qb = draft_probs + (size_t)b * K * (size_t)V;
    const float* pb = target_probs + (size_t)b * (K + 1) * (size_t)V;
    /* w_0 .. w_K */
    float w[65];
    if (K > 64) return -1;
    w[0] = 1.0f;
    for (int k = 0; k < K; ++k) {
      int d = tokens[(size_t)b * K + k];
      if (d < 0 || d >= V) return -1;
      float ratio = pb[(size_t)k * V + d] / qb[(size_t)k * V + d];
      float t = w[k] * ratio;
      w[k + 1] = t < 1.0f ? t : (t >= 1.0f ? 1.0f : 0.0f); /* NaN -> 0 */
    }
    int tau = 0;
    for (int i = 1; i <= K; ++i) {
      double h;
      if (i < K) {
        const float* p = pb + (size_t)i * V;
        const float* q = qb + (size_t)i * V;
        double r = 0.0;
        for (int x = 0; x < V; ++x) {
          float term = w[i] * p[x] - q[x];
          if (term > 0.0f) r += (double)term;
        }
        double den = r + (1.0 - (double)w[i]);
        h = den > 0.0 ? r / den : 1.0;
      } else {
        h = (double)w[K];
      }
      float eta = oracle_accept_uniform(
          oracle_noise_word(seed[b], offset[b], i - 1, 1, 0u));
      if ((double)eta <= h) tau = i;
      if (h_out) h_out[(size_t)b * K + (i - 1)] = h;
      if (eta_out) eta_out[(size_t)b * K + (i - 1)] = eta;
    }
    int emit;
    float best = -INFINITY, second = -INFINITY;
    const float* p = pb + (size_t)tau * V;
    if (tau == K) {
      emit = gumbel_max_weights(p, V, seed[b], offset[b], K, &best, &second);
    } else {
      const float* q = qb + (size_t)tau * V;
      int any = 0;
      for (int x = 0; x < V; ++x) {
        float term = w[tau] * p[x] - q[x];
        residual_scratch[x] = term > 0.0f ? term : 0.0f;
        if (residual_scratch[x] > 0.0f) any = 1;
      }
      emit = gumbel_max_weights(any ? residual_scratch : p, V, seed[b],
                                offset[b], tau, &best, &second);
    }
    accepted_len[b] = tau;
    emitted[b] = emit < 0 ? 0 : emit;
    if (emit_top2) {
      emit_top2[2 * b] = best;
      emit_top2[2 * b + 1] = second;
    }
  }
  return 0;
}

/* ------------------------------------------ temperature-only target sampler */

/*
 * Temperature-only sampling of target rows: PR #27, "1. Temperature-only
 * sampling runs no filter" (softmax and sampling only, no top-k, top-p or
 * min-p).  Row i of logits [R,V] (float32) is drawn like a draft position
 * (oracle_sample_row): s = l / T_i, token = argmax of float(s + g) with g
 * from noise stream 3 at position position[i] (argmax of s for a greedy
 * row), probs = softmax(s) in double (one-hot for greedy).  T [R]: the rows'
 * temperatures (finite and > 0); greedy, position: [R] or NULL (0).
 * probs [R,V] double, rowstats [R,2] (M, S) and top2 [R,2] may be NULL.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_sample_temperature(const float* logits, const float* T,
                              const uint8_t* greedy, const uint64_t* seed,
                              const uint64_t* offset, const int32_t* position,
                              int R, int V, int32_t* tokens, double* probs,
                              double* rowstats, float* top2,
                              double* probs_scratch) {
  if (R <= 0 || V <= 0 || !logits || !T || !seed || !offset || !tokens ||
      !probs_scratch)
    return -1;
  for (int i = 0; i < R; ++i) {
    if (!(T[i] > 0.0f) || !isfinite(T[i])) return -1;
    int pos = position ? position[i] : 0;
    if (pos < 0 || pos > 0xffff) return -1;
    double* q = probs ? probs + (size_t)i * V : probs_scratch;
    int token;
    double M, S;
    float best, second;
    oracle_sample_row(logits + (size_t)i * V, V, seed[i], offset[i], pos, 3,
                      T[i], greedy ? greedy[i] != 0 : 0, q, &token, &M, &S,
                      &best, &second);
    tokens[i] = token;
    if (rowstats) {
      rowstats[2 * i] = M;
      rowstats[2 * i + 1] = S;
    }
    if (top2) {
      top2[2 * i] = best;
      top2[2 * i + 1] = second;
    }
  }
  return 0;
}
