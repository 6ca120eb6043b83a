/*
 * gdn_oracle.c -- double-precision CPU oracle for speculative verify and
 * replay commit of Gated DeltaNet (GDN) layers.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load or call this file.  It shares no source, header,
 * table or helper with the CUDA library; the two only meet through arrays the
 * seeded input generator builds.
 *
 * Everything here is plain loops in fp64, one token at a time, in the order
 * the method states it.  The only parallelism is OpenMP over independent
 * (row, head) or (layer, row) units; no arithmetic is blocked, fused or
 * reordered.
 *
 * What is computed (state S is one [V][K] matrix per value head, row-major,
 * K contiguous):
 *   alpha_t = exp(-exp(A_log) * softplus(a_t + dt_bias))   the decay exp(g)
 *   beta_t  = sigmoid(b_t)
 *   khat_t  = k_t / sqrt(|k_t|^2 + eps),  qhat_t likewise  (eps = 1e-6)
 *   H       = alpha_t * S_{t-1}
 *   u_t     = beta_t * (v_t - H khat_t)                   the correction
 *   S_t     = H + u_t khat_t^T
 *   o_t     = S_t qhat_t
 * Sources: the per-token replay record [correction (V), normalized key (K),
 * gate (1)] is listed in vLLM PR "[Spec Decode][Qwen4Exp] RecoverSSM for
 * Qwen GDN and the PLE short conv", Purpose; the forward update
 * h = fma(c, k, h * decay) with decay exp(g) in the same PR, Test Result
 * (Output bullet); the per-value-head [V,K] state in lmdeploy PR "opt-in
 * ReplaySSM", Copilot review findings.  The gate formulas and the delta-rule
 * correction are the standard Gated DeltaNet recurrence.
 *
 * Parity: pinned by tests/test_oracle_pins.py (closed forms, a hand-worked
 * two-token example in tests/golden/, invariants and a brute-force plan
 * enumeration).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Row error bits, as documented for the library's optional error word. */
#define ORACLE_ERR_WINDOW   1  /* window_len outside [0, max_window]            */
#define ORACLE_ERR_ACCEPTED 2  /* accepted_len outside [0, window_len]           */
#define ORACLE_ERR_SLOT     4  /* slot outside [-1, num_slots)                   */
#define ORACLE_ERR_BLOCK    8  /* align mode: referenced column outside table,  */
                               /* or -1 where a live row needs a slot            */
#define ORACLE_ERR_SEQPOS  16  /* align mode: seq_pos < 1                        */
#define ORACLE_ERR_TOKENS  32  /* token rows outside [0, num_tokens)             */

static const double L2NORM_EPS = 1e-6;

int gdn_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads the parallel loops use from now on (the benchmark times the
 * oracle on all host cores and on one). */
void gdn_oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* softplus(x) = log(1 + e^x), written so that neither branch overflows. */
double gdn_oracle_softplus(double x) {
  if (x > 0.0) return x + log1p(exp(-x));
  return log1p(exp(x));
}

/* The decay the verify records, alpha = exp(g) with
 * g = -exp(A_log) * softplus(a + dt_bias). */
double gdn_oracle_decay(double a, double A_log, double dt_bias) {
  double g = -exp(A_log) * gdn_oracle_softplus(a + dt_bias);
  return exp(g);
}

/* The write strength beta = sigmoid(b). */
double gdn_oracle_beta(double b) { return 1.0 / (1.0 + exp(-b)); }

/* out = x / sqrt(sum(x^2) + eps). */
void gdn_oracle_l2norm(int n, const double* x, double* out) {
  double ss = 0.0;
  for (int j = 0; j < n; ++j) ss += x[j] * x[j];
  double norm = sqrt(ss + L2NORM_EPS);
  for (int j = 0; j < n; ++j) out[j] = x[j] / norm;
}

/* One token of the gated delta rule on S[V][K], in place.
 * u_out[V] receives the correction, o_out[V] the output. */
static void token_step(int K, int V, double* S, const double* khat,
                       const double* qhat, const double* v, double alpha,
                       double beta, double* u_out, double* o_out) {
  /* H = alpha * S */
  for (int i = 0; i < V; ++i)
    for (int j = 0; j < K; ++j) S[(size_t)i * K + j] *= alpha;
  /* u = beta * (v - H khat) */
  for (int i = 0; i < V; ++i) {
    double d = 0.0;
    for (int j = 0; j < K; ++j) d += S[(size_t)i * K + j] * khat[j];
    u_out[i] = beta * (v[i] - d);
  }
  /* S = H + u khat^T */
  for (int i = 0; i < V; ++i)
    for (int j = 0; j < K; ++j) S[(size_t)i * K + j] += u_out[i] * khat[j];
  /* o = S qhat */
  for (int i = 0; i < V; ++i) {
    double o = 0.0;
    for (int j = 0; j < K; ++j) o += S[(size_t)i * K + j] * qhat[j];
    o_out[i] = o;
  }
}

/* The verify window of one (request, value head) unit.
 *   S0      [V*K]  checkpoint state (read only)
 *   q, k    [w][K] raw query / key rows for this unit's key head
 *   v       [w][V] value rows for this value head
 *   a, b    [w]    raw gate inputs
 * Outputs (any may be NULL): o [w][V], u [w][V], khat [w][K], alpha [w],
 * states [w][V*K] = state after each token.  Nothing is written to S0:
 * the verify runs from a read-only checkpoint. */
void gdn_oracle_window(int K, int V, int w, const double* S0, const double* q,
                       const double* k, const double* v, const double* a,
                       const double* b, double A_log, double dt_bias,
                       double* o, double* u, double* khat, double* alpha,
                       double* states) {
  size_t VK = (size_t)V * K;
  double* S = (double*)malloc(VK * sizeof(double));
  double* kh = (double*)malloc((size_t)K * sizeof(double));
  double* qh = (double*)malloc((size_t)K * sizeof(double));
  double* ut = (double*)malloc((size_t)V * sizeof(double));
  double* ot = (double*)malloc((size_t)V * sizeof(double));
  memcpy(S, S0, VK * sizeof(double));
  for (int t = 0; t < w; ++t) {
    double al = gdn_oracle_decay(a[t], A_log, dt_bias);
    double be = gdn_oracle_beta(b[t]);
    gdn_oracle_l2norm(K, k + (size_t)t * K, kh);
    gdn_oracle_l2norm(K, q + (size_t)t * K, qh);
    token_step(K, V, S, kh, qh, v + (size_t)t * V, al, be, ut, ot);
    if (o) memcpy(o + (size_t)t * V, ot, (size_t)V * sizeof(double));
    if (u) memcpy(u + (size_t)t * V, ut, (size_t)V * sizeof(double));
    if (khat) memcpy(khat + (size_t)t * K, kh, (size_t)K * sizeof(double));
    if (alpha) alpha[t] = al;
    if (states) memcpy(states + (size_t)t * VK, S, VK * sizeof(double));
  }
  free(S); free(kh); free(qh); free(ut); free(ot);
}

/* Forward replay of n recorded tokens on S[V][K], in place:
 * S = alpha_t * S + u_t khat_t^T for t = 0..n-1 (the commit's fold). */
void gdn_oracle_replay(int K, int V, int n, double* S, const double* u,
                       const double* khat, const double* alpha) {
  for (int t = 0; t < n; ++t) {
    const double* ut = u + (size_t)t * V;
    const double* kt = khat + (size_t)t * K;
    for (int i = 0; i < V; ++i)
      for (int j = 0; j < K; ++j) {
        double h = S[(size_t)i * K + j] * alpha[t];
        S[(size_t)i * K + j] = h + ut[i] * kt[j];
      }
  }
}

/* Slot that holds the state after x folded tokens of row `table_row`.
 * Without align mode (block_size == 0) a request owns one slot, column 0.
 * In align mode the state after x tokens lives in the block of its last
 * token, column (x - 1) / block_size (vLLM PR above, Commits item 3).
 * Returns OUTSIDE_TABLE if the column lies outside the table. */
#define OUTSIDE_TABLE INT32_MIN
static int32_t slot_after(const int32_t* table_row, int table_stride,
                          int block_size, long x) {
  if (block_size == 0) return table_row[0];
  long col = (x - 1) / block_size;
  if (x < 1 || col >= table_stride) return OUTSIDE_TABLE;
  return table_row[col];
}

/* Source slot of a row's verify: the checkpoint after seq_pos tokens.
 * An empty window reads nothing and counts as a null row (-1).
 * Returns the slot (>= -1) or a negative error: -(1 + error bits). */
int gdn_oracle_source_slot(int window_len, const int32_t* table_row,
                           int table_stride, int seq_pos, int block_size,
                           int num_slots, int max_window) {
  if (window_len < 0 || window_len > max_window)
    return -(1 + ORACLE_ERR_WINDOW);
  if (window_len == 0) return -1;
  if (block_size > 0 && seq_pos < 1) return -(1 + ORACLE_ERR_SEQPOS);
  int32_t s = slot_after(table_row, table_stride, block_size, seq_pos);
  if (s == OUTSIDE_TABLE) return -(1 + ORACLE_ERR_BLOCK);
  if (s < -1 || s >= num_slots) return -(1 + ORACLE_ERR_SLOT);
  return s;
}

/* Commit plan of one row: which slots receive the state after how many
 * accepted tokens.  The final state after n = accepted_len tokens goes to
 * slot(p0 + n); in align mode every block boundary p strictly inside
 * (p0, p0 + n) -- p a multiple of block_size -- also stores the state after
 * p - p0 tokens into slot(p).  A boundary at p0 + n is the final state
 * itself and is not written twice.  Rows with a null source slot (-1) or
 * n == 0 write nothing (vLLM PR above, Purpose: graph padding rows;
 * Commits items 3 and 6).
 * Returns the number of writes (final first), or -(1 + error bits). */
int gdn_oracle_commit_plan(int window_len, int accepted_len,
                           const int32_t* table_row, int table_stride,
                           int seq_pos, int block_size, int num_slots,
                           int max_window, int32_t* src_slot,
                           int32_t* out_slot, int32_t* out_ntok,
                           int max_writes) {
  int src = gdn_oracle_source_slot(window_len, table_row, table_stride,
                                   seq_pos, block_size, num_slots, max_window);
  if (src < -1) return src;
  if (accepted_len < 0 || accepted_len > window_len)
    return -(1 + ORACLE_ERR_ACCEPTED);
  *src_slot = src;
  if (src == -1 || accepted_len == 0) return 0;
  long p0 = block_size > 0 ? seq_pos : 0;
  int n = accepted_len;
  int nw = 0;
  int32_t fin = slot_after(table_row, table_stride, block_size, p0 + n);
  if (fin == OUTSIDE_TABLE || fin == -1) return -(1 + ORACLE_ERR_BLOCK);
  if (fin < -1 || fin >= num_slots) return -(1 + ORACLE_ERR_SLOT);
  if (nw < max_writes) { out_slot[nw] = fin; out_ntok[nw] = n; }
  ++nw;
  if (block_size > 0) {
    for (long p = p0 + 1; p < p0 + n; ++p) {
      if (p % block_size != 0) continue;
      int32_t s = slot_after(table_row, table_stride, block_size, p);
      if (s == OUTSIDE_TABLE || s == -1) return -(1 + ORACLE_ERR_BLOCK);
      if (s < -1 || s >= num_slots) return -(1 + ORACLE_ERR_SLOT);
      if (nw < max_writes) { out_slot[nw] = s; out_ntok[nw] = (int32_t)(p - p0); }
      ++nw;
    }
  }
  return nw;
}

/* Verify (and, when snaps != NULL, the native per-draft snapshots) for all
 * rows of one layer.
 *   q, k  [T][HK][K]; v [T][HV][V]; a, b [T][HV]; A_log, dt_bias [HV]
 *   token_start[B], window_len[B]: row b owns token rows
 *       token_start[b] .. token_start[b] + window_len[b] - 1
 *   pool  [num_slots][HV][V][K] (read only)
 *   out   [T][HV][V]; rec_u [B][HV][W_max][V]; rec_k [B][HV][W_max][K];
 *   rec_g [B][HV][W_max]; snaps [B][W_max][HV][V][K] (optional)
 *   row_err[B] receives the row's error bits (0 if fine).
 * Value head h reads key head h / (HV / HK).  Rows that are malformed, have
 * a null slot or an empty window write nothing. */
int gdn_oracle_spec_verify(int HK, int HV, int K, int V, int W_max, int B,
                           int T, int num_slots, const double* q,
                           const double* k, const double* v, const double* a,
                           const double* b, const double* A_log,
                           const double* dt_bias, const int32_t* token_start,
                           const int32_t* window_len, const double* pool,
                           const int32_t* slot_table, int table_stride,
                           const int32_t* seq_pos, int block_size,
                           double* out, double* rec_u, double* rec_k,
                           double* rec_g, double* snaps, int32_t* row_err) {
  if (HK <= 0 || HV <= 0 || HV % HK != 0 || K <= 0 || V <= 0 || W_max <= 0)
    return -2;
  int group = HV / HK;
  size_t VK = (size_t)V * K;
  for (int r = 0; r < B; ++r) row_err[r] = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long unit = 0; unit < (long)B * HV; ++unit) {
    int r = (int)(unit / HV), h = (int)(unit % HV);
    int w = window_len[r];
    int sp = seq_pos ? seq_pos[r] : 0;
    int src = gdn_oracle_source_slot(w, slot_table + (size_t)r * table_stride,
                                     table_stride, sp, block_size, num_slots,
                                     W_max);
    int err = src < -1 ? -src - 1 : 0;
    long t0 = token_start[r];
    if (!err && w > 0 && src >= 0 && (t0 < 0 || t0 + w > T))
      err = ORACLE_ERR_TOKENS;
    if (err) { if (h == 0) row_err[r] = err; continue; }
    if (src < 0 || w == 0) continue;
    int hk = h / group;
    double* qa = (double*)malloc((size_t)w * K * sizeof(double));
    double* ka = (double*)malloc((size_t)w * K * sizeof(double));
    double* va = (double*)malloc((size_t)w * V * sizeof(double));
    double* aa = (double*)malloc((size_t)w * sizeof(double));
    double* ba = (double*)malloc((size_t)w * sizeof(double));
    double* oa = (double*)malloc((size_t)w * V * sizeof(double));
    double* ua = (double*)malloc((size_t)w * V * sizeof(double));
    double* kh = (double*)malloc((size_t)w * K * sizeof(double));
    double* ga = (double*)malloc((size_t)w * sizeof(double));
    double* st = snaps ? (double*)malloc((size_t)w * VK * sizeof(double)) : NULL;
    for (int t = 0; t < w; ++t) {
      long row = t0 + t;
      memcpy(qa + (size_t)t * K, q + ((size_t)row * HK + hk) * K, (size_t)K * sizeof(double));
      memcpy(ka + (size_t)t * K, k + ((size_t)row * HK + hk) * K, (size_t)K * sizeof(double));
      memcpy(va + (size_t)t * V, v + ((size_t)row * HV + h) * V, (size_t)V * sizeof(double));
      aa[t] = a[(size_t)row * HV + h];
      ba[t] = b[(size_t)row * HV + h];
    }
    const double* S0 = pool + ((size_t)src * HV + h) * VK;
    gdn_oracle_window(K, V, w, S0, qa, ka, va, aa, ba, A_log[h], dt_bias[h],
                      oa, ua, kh, ga, st);
    for (int t = 0; t < w; ++t) {
      long row = t0 + t;
      if (out)
        memcpy(out + ((size_t)row * HV + h) * V, oa + (size_t)t * V, (size_t)V * sizeof(double));
      size_t rec = ((size_t)r * HV + h) * W_max + t;
      if (rec_u) memcpy(rec_u + rec * V, ua + (size_t)t * V, (size_t)V * sizeof(double));
      if (rec_k) memcpy(rec_k + rec * K, kh + (size_t)t * K, (size_t)K * sizeof(double));
      if (rec_g) rec_g[rec] = ga[t];
      if (snaps)
        memcpy(snaps + (((size_t)r * W_max + t) * HV + h) * VK, st + (size_t)t * VK,
               VK * sizeof(double));
    }
    free(qa); free(ka); free(va); free(aa); free(ba);
    free(oa); free(ua); free(kh); free(ga); free(st);
  }
  return 0;
}

/* All-layer replay commit from records, with layers in KV-cache groups.
 *   pools_in  [L][num_slots][HV][V][K]  states before the commit (read only)
 *   pools_out [L][num_slots][HV][V][K]  the caller's copy of pools_in; the
 *             planned slots are overwritten.  Reading every fold's source
 *             from pools_in makes the result independent of write order,
 *             which is what running final folds before boundary folds
 *             guarantees on the GPU (vLLM PR above, Commits item 6).
 *   rec_u [L][B][HV][W_max][V], rec_k [L][B][HV][W_max][K],
 *   rec_g [L][B][HV][W_max]
 *   layer_group [L]: group of each layer (NULL: every layer in group 0);
 *   group g's slot table starts at slot_table + g * group_stride (the
 *   [group, batch] state-index table of the vLLM PR's review thread).
 *   row_err[B] receives the row's error bits, OR-ed over the groups. */
int gdn_oracle_replay_commit_grouped(int L, int HV, int K, int V, int W_max,
                                     int B, int num_slots,
                                     const double* pools_in, double* pools_out,
                                     const double* rec_u, const double* rec_k,
                                     const double* rec_g,
                                     const int32_t* window_len,
                                     const int32_t* accepted_len,
                                     const int32_t* layer_group,
                                     int num_groups, long group_stride,
                                     const int32_t* slot_table,
                                     int table_stride, const int32_t* seq_pos,
                                     int block_size, int32_t* row_err) {
  if (L <= 0 || HV <= 0 || K <= 0 || V <= 0 || W_max <= 0 || num_groups <= 0)
    return -2;
  if (layer_group)
    for (int l = 0; l < L; ++l)
      if (layer_group[l] < 0 || layer_group[l] >= num_groups) return -3;
  size_t VK = (size_t)V * K;
  size_t pool_elems = (size_t)num_slots * HV * VK;
  int max_writes = 2 + W_max;
  for (int r = 0; r < B; ++r) row_err[r] = 0;
  for (int g = 0; g < num_groups; ++g) {
    for (int r = 0; r < B; ++r) {
      int32_t src, slots[64], ntok[64];
      int sp = seq_pos ? seq_pos[r] : 0;
      const int32_t* trow = slot_table + g * group_stride + (size_t)r * table_stride;
      int nw = gdn_oracle_commit_plan(window_len[r], accepted_len[r], trow,
                                      table_stride, sp, block_size, num_slots,
                                      W_max, &src, slots, ntok, max_writes);
      if (nw < 0) row_err[r] |= -nw - 1;
    }
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (long unit = 0; unit < (long)L * B * HV; ++unit) {
    int l = (int)(unit / ((long)B * HV));
    int r = (int)((unit / HV) % B);
    int h = (int)(unit % HV);
    int g = layer_group ? layer_group[l] : 0;
    int32_t src, slots[64], ntok[64];
    int sp = seq_pos ? seq_pos[r] : 0;
    const int32_t* trow = slot_table + g * group_stride + (size_t)r * table_stride;
    int nw = gdn_oracle_commit_plan(window_len[r], accepted_len[r], trow,
                                    table_stride, sp, block_size, num_slots,
                                    W_max, &src, slots, ntok, max_writes);
    if (nw <= 0) continue;
    size_t rec = (((size_t)l * B + r) * HV + h) * W_max;
    double* S = (double*)malloc(VK * sizeof(double));
    for (int i = 0; i < nw; ++i) {
      memcpy(S, pools_in + l * pool_elems + ((size_t)src * HV + h) * VK,
             VK * sizeof(double));
      gdn_oracle_replay(K, V, ntok[i], S, rec_u + rec * V, rec_k + rec * K,
                        rec_g + rec);
      memcpy(pools_out + l * pool_elems + ((size_t)slots[i] * HV + h) * VK, S,
             VK * sizeof(double));
    }
    free(S);
  }
  return 0;
}

/* All-layer replay commit with every layer reading the same slot table. */
int gdn_oracle_replay_commit(int L, int HV, int K, int V, int W_max, int B,
                             int num_slots, const double* pools_in,
                             double* pools_out, const double* rec_u,
                             const double* rec_k, const double* rec_g,
                             const int32_t* window_len,
                             const int32_t* accepted_len,
                             const int32_t* slot_table, int table_stride,
                             const int32_t* seq_pos, int block_size,
                             int32_t* row_err) {
  return gdn_oracle_replay_commit_grouped(
      L, HV, K, V, W_max, B, num_slots, pools_in, pools_out, rec_u, rec_k,
      rec_g, window_len, accepted_len, NULL, 1, 0, slot_table, table_stride,
      seq_pos, block_size, row_err);
}

/* Short-conv state commit (vLLM PR above, Purpose: the conv state advances
 * over the accepted tokens by the recurrent commit's plan).  A layer's causal depthwise
 * convolution of width SL + 1 keeps, per slot and channel, the last SL
 * convolution inputs, oldest first: state [C][SL].  The state after x
 * folded tokens of a row is the last SL entries of
 *     (checkpoint state of the channel) ++ (the row's first x window inputs),
 * written to the slots the SSM commit plan names for x tokens.
 *   pools_in / pools_out [L][num_slots][C][SL]   (pools_out: caller's copy)
 *   inputs [L][T][C]: convolution inputs of every token row
 *   token_start[B]: first token row of each request's window
 * Row errors are the commit plan's, then GDN_ROW_ERR_TOKENS when a live
 * row's window rows fall outside [0, T). */
int gdn_oracle_conv_commit(int L, int C, int SL, int W_max, int B, int T,
                           int num_slots, const double* pools_in,
                           double* pools_out, const double* inputs,
                           const int32_t* token_start,
                           const int32_t* window_len,
                           const int32_t* accepted_len,
                           const int32_t* layer_group, int num_groups,
                           long group_stride, const int32_t* slot_table,
                           int table_stride, const int32_t* seq_pos,
                           int block_size, int32_t* row_err) {
  if (L <= 0 || C <= 0 || SL <= 0 || W_max <= 0 || num_groups <= 0) return -2;
  if (layer_group)
    for (int l = 0; l < L; ++l)
      if (layer_group[l] < 0 || layer_group[l] >= num_groups) return -3;
  size_t pool_elems = (size_t)num_slots * C * SL;
  int max_writes = 2 + W_max;
  for (int r = 0; r < B; ++r) row_err[r] = 0;
  double* seq = (double*)malloc((size_t)(SL + W_max) * sizeof(double));
  for (int l = 0; l < L; ++l) {
    int g = layer_group ? layer_group[l] : 0;
    for (int r = 0; r < B; ++r) {
      int32_t src, slots[64], ntok[64];
      int sp = seq_pos ? seq_pos[r] : 0;
      const int32_t* trow = slot_table + g * group_stride + (size_t)r * table_stride;
      int nw = gdn_oracle_commit_plan(window_len[r], accepted_len[r], trow,
                                      table_stride, sp, block_size, num_slots,
                                      W_max, &src, slots, ntok, max_writes);
      if (nw < 0) { row_err[r] |= -nw - 1; continue; }
      if (nw == 0) continue;
      long t0 = token_start[r];
      if (t0 < 0 || t0 + window_len[r] > T) { row_err[r] |= ORACLE_ERR_TOKENS; continue; }
      for (int c = 0; c < C; ++c) {
        const double* old = pools_in + l * pool_elems + ((size_t)src * C + c) * SL;
        for (int j = 0; j < SL; ++j) seq[j] = old[j];
        for (int i = 0; i < accepted_len[r]; ++i)
          seq[SL + i] = inputs[((size_t)l * T + t0 + i) * C + c];
        for (int w = 0; w < nw; ++w) {
          double* dst = pools_out + l * pool_elems + ((size_t)slots[w] * C + c) * SL;
          for (int j = 0; j < SL; ++j) dst[j] = seq[ntok[w] + j];
        }
      }
    }
  }
  free(seq);
  return 0;
}

/* ------------------------------------------------------------------ KDA
 * Per-channel decay (KDA, the Kimi Delta Attention layer the protocol was
 * first built for: tokenspeed PR "feat: add Qwen3.5 GDN ReplaySSM",
 * Summary; vLLM PR above, Purpose).  The pages print no KDA formula; the
 * reading taken here replaces the scalar decay of the gated delta rule by a
 * vector over the K key channels, everything else unchanged:
 *   alpha_t[j] = exp(-exp(A_log) * softplus(a_t[j] + dt_bias[j])),  j < K
 *   H          = S_{t-1} diag(alpha_t)   (column j of S scaled by alpha_t[j])
 *   u_t        = beta_t * (v_t - H khat_t)
 *   S_t        = H + u_t khat_t^T
 *   o_t        = S_t qhat_t
 * and the replay record keeps the whole gate vector: (u_t, khat_t, alpha_t
 * in R^K).  The commit's fold is S = alpha_t-scaled columns plus the
 * rank-one write, token by token. */

/* One KDA token on S[V][K], in place; alpha[K] is the gate vector. */
static void kda_token_step(int K, int V, double* S, const double* khat,
                           const double* qhat, const double* v,
                           const double* alpha, double beta, double* u_out,
                           double* o_out) {
  /* H = S diag(alpha): every element of column j scaled by alpha[j] */
  for (int i = 0; i < V; ++i)
    for (int j = 0; j < K; ++j) S[(size_t)i * K + j] *= alpha[j];
  /* u = beta * (v - H khat) */
  for (int i = 0; i < V; ++i) {
    double d = 0.0;
    for (int j = 0; j < K; ++j) d += S[(size_t)i * K + j] * khat[j];
    u_out[i] = beta * (v[i] - d);
  }
  /* S = H + u khat^T */
  for (int i = 0; i < V; ++i)
    for (int j = 0; j < K; ++j) S[(size_t)i * K + j] += u_out[i] * khat[j];
  /* o = S qhat */
  for (int i = 0; i < V; ++i) {
    double o = 0.0;
    for (int j = 0; j < K; ++j) o += S[(size_t)i * K + j] * qhat[j];
    o_out[i] = o;
  }
}

/* The KDA verify window of one (request, value head) unit.
 *   a [w][K] raw per-channel gate inputs, dt_bias [K]; otherwise as
 *   gdn_oracle_window.  alpha (optional) receives [w][K] gate vectors. */
void gdn_oracle_kda_window(int K, int V, int w, const double* S0,
                           const double* q, const double* k, const double* v,
                           const double* a, const double* b, double A_log,
                           const double* dt_bias, double* o, double* u,
                           double* khat, double* alpha, double* states) {
  size_t VK = (size_t)V * K;
  double* S = (double*)malloc(VK * sizeof(double));
  double* kh = (double*)malloc((size_t)K * sizeof(double));
  double* qh = (double*)malloc((size_t)K * sizeof(double));
  double* al = (double*)malloc((size_t)K * sizeof(double));
  double* ut = (double*)malloc((size_t)V * sizeof(double));
  double* ot = (double*)malloc((size_t)V * sizeof(double));
  memcpy(S, S0, VK * sizeof(double));
  for (int t = 0; t < w; ++t) {
    for (int j = 0; j < K; ++j)
      al[j] = gdn_oracle_decay(a[(size_t)t * K + j], A_log, dt_bias[j]);
    double be = gdn_oracle_beta(b[t]);
    gdn_oracle_l2norm(K, k + (size_t)t * K, kh);
    gdn_oracle_l2norm(K, q + (size_t)t * K, qh);
    kda_token_step(K, V, S, kh, qh, v + (size_t)t * V, al, be, ut, ot);
    if (o) memcpy(o + (size_t)t * V, ot, (size_t)V * sizeof(double));
    if (u) memcpy(u + (size_t)t * V, ut, (size_t)V * sizeof(double));
    if (khat) memcpy(khat + (size_t)t * K, kh, (size_t)K * sizeof(double));
    if (alpha) memcpy(alpha + (size_t)t * K, al, (size_t)K * sizeof(double));
    if (states) memcpy(states + (size_t)t * VK, S, VK * sizeof(double));
  }
  free(S); free(kh); free(qh); free(al); free(ut); free(ot);
}

/* Forward replay of n recorded KDA tokens on S[V][K], in place:
 * S[i][j] = alpha_t[j] * S[i][j] + u_t[i] khat_t[j], t = 0..n-1. */
void gdn_oracle_kda_replay(int K, int V, int n, double* S, const double* u,
                           const double* khat, const double* alpha) {
  for (int t = 0; t < n; ++t) {
    const double* ut = u + (size_t)t * V;
    const double* kt = khat + (size_t)t * K;
    const double* at = alpha + (size_t)t * K;
    for (int i = 0; i < V; ++i)
      for (int j = 0; j < K; ++j) {
        double h = S[(size_t)i * K + j] * at[j];
        S[(size_t)i * K + j] = h + ut[i] * kt[j];
      }
  }
}

/* KDA verify (and, when snaps != NULL, native snapshots) of one layer.
 * As gdn_oracle_spec_verify, except a [T][HV][K], dt_bias [HV][K] and
 * rec_g [B][HV][W_max][K]. */
int gdn_oracle_kda_spec_verify(int HK, int HV, int K, int V, int W_max, int B,
                               int T, int num_slots, const double* q,
                               const double* k, const double* v,
                               const double* a, const double* b,
                               const double* A_log, const double* dt_bias,
                               const int32_t* token_start,
                               const int32_t* window_len, const double* pool,
                               const int32_t* slot_table, int table_stride,
                               const int32_t* seq_pos, int block_size,
                               double* out, double* rec_u, double* rec_k,
                               double* rec_g, double* snaps, int32_t* row_err) {
  if (HK <= 0 || HV <= 0 || HV % HK != 0 || K <= 0 || V <= 0 || W_max <= 0)
    return -2;
  int group = HV / HK;
  size_t VK = (size_t)V * K;
  for (int r = 0; r < B; ++r) row_err[r] = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long unit = 0; unit < (long)B * HV; ++unit) {
    int r = (int)(unit / HV), h = (int)(unit % HV);
    int w = window_len[r];
    int sp = seq_pos ? seq_pos[r] : 0;
    int src = gdn_oracle_source_slot(w, slot_table + (size_t)r * table_stride,
                                     table_stride, sp, block_size, num_slots,
                                     W_max);
    int err = src < -1 ? -src - 1 : 0;
    long t0 = token_start[r];
    if (!err && w > 0 && src >= 0 && (t0 < 0 || t0 + w > T))
      err = ORACLE_ERR_TOKENS;
    if (err) { if (h == 0) row_err[r] = err; continue; }
    if (src < 0 || w == 0) continue;
    int hk = h / group;
    double* qa = (double*)malloc((size_t)w * K * sizeof(double));
    double* ka = (double*)malloc((size_t)w * K * sizeof(double));
    double* va = (double*)malloc((size_t)w * V * sizeof(double));
    double* aa = (double*)malloc((size_t)w * K * sizeof(double));
    double* ba = (double*)malloc((size_t)w * sizeof(double));
    double* oa = (double*)malloc((size_t)w * V * sizeof(double));
    double* ua = (double*)malloc((size_t)w * V * sizeof(double));
    double* kh = (double*)malloc((size_t)w * K * sizeof(double));
    double* ga = (double*)malloc((size_t)w * K * sizeof(double));
    double* st = snaps ? (double*)malloc((size_t)w * VK * sizeof(double)) : NULL;
    for (int t = 0; t < w; ++t) {
      long row = t0 + t;
      memcpy(qa + (size_t)t * K, q + ((size_t)row * HK + hk) * K, (size_t)K * sizeof(double));
      memcpy(ka + (size_t)t * K, k + ((size_t)row * HK + hk) * K, (size_t)K * sizeof(double));
      memcpy(va + (size_t)t * V, v + ((size_t)row * HV + h) * V, (size_t)V * sizeof(double));
      memcpy(aa + (size_t)t * K, a + ((size_t)row * HV + h) * K, (size_t)K * sizeof(double));
      ba[t] = b[(size_t)row * HV + h];
    }
    const double* S0 = pool + ((size_t)src * HV + h) * VK;
    gdn_oracle_kda_window(K, V, w, S0, qa, ka, va, aa, ba, A_log[h],
                          dt_bias + (size_t)h * K, oa, ua, kh, ga, st);
    for (int t = 0; t < w; ++t) {
      long row = t0 + t;
      if (out)
        memcpy(out + ((size_t)row * HV + h) * V, oa + (size_t)t * V, (size_t)V * sizeof(double));
      size_t rec = ((size_t)r * HV + h) * W_max + t;
      if (rec_u) memcpy(rec_u + rec * V, ua + (size_t)t * V, (size_t)V * sizeof(double));
      if (rec_k) memcpy(rec_k + rec * K, kh + (size_t)t * K, (size_t)K * sizeof(double));
      if (rec_g) memcpy(rec_g + rec * K, ga + (size_t)t * K, (size_t)K * sizeof(double));
      if (snaps)
        memcpy(snaps + (((size_t)r * W_max + t) * HV + h) * VK, st + (size_t)t * VK,
               VK * sizeof(double));
    }
    free(qa); free(ka); free(va); free(aa); free(ba);
    free(oa); free(ua); free(kh); free(ga); free(st);
  }
  return 0;
}

/* All-layer KDA replay commit from records (one slot table for every
 * layer).  As gdn_oracle_replay_commit, except rec_g [L][B][HV][W_max][K]:
 * every fold reads its source from pools_in, so the result does not depend
 * on the order of the writes. */
int gdn_oracle_kda_replay_commit(int L, int HV, int K, int V, int W_max, int B,
                                 int num_slots, const double* pools_in,
                                 double* pools_out, const double* rec_u,
                                 const double* rec_k, const double* rec_g,
                                 const int32_t* window_len,
                                 const int32_t* accepted_len,
                                 const int32_t* slot_table, int table_stride,
                                 const int32_t* seq_pos, int block_size,
                                 int32_t* row_err) {
  if (L <= 0 || HV <= 0 || K <= 0 || V <= 0 || W_max <= 0) return -2;
  size_t VK = (size_t)V * K;
  size_t pool_elems = (size_t)num_slots * HV * VK;
  int max_writes = 2 + W_max;
  for (int r = 0; r < B; ++r) {
    int32_t src, slots[64], ntok[64];
    int sp = seq_pos ? seq_pos[r] : 0;
    int nw = gdn_oracle_commit_plan(window_len[r], accepted_len[r],
                                    slot_table + (size_t)r * table_stride,
                                    table_stride, sp, block_size, num_slots,
                                    W_max, &src, slots, ntok, max_writes);
    row_err[r] = nw < 0 ? -nw - 1 : 0;
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (long unit = 0; unit < (long)L * B * HV; ++unit) {
    int l = (int)(unit / ((long)B * HV));
    int r = (int)((unit / HV) % B);
    int h = (int)(unit % HV);
    int32_t src, slots[64], ntok[64];
    int sp = seq_pos ? seq_pos[r] : 0;
    int nw = gdn_oracle_commit_plan(window_len[r], accepted_len[r],
                                    slot_table + (size_t)r * table_stride,
                                    table_stride, sp, block_size, num_slots,
                                    W_max, &src, slots, ntok, max_writes);
    if (nw <= 0) continue;
    size_t rec = (((size_t)l * B + r) * HV + h) * W_max;
    double* S = (double*)malloc(VK * sizeof(double));
    for (int i = 0; i < nw; ++i) {
      memcpy(S, pools_in + l * pool_elems + ((size_t)src * HV + h) * VK,
             VK * sizeof(double));
      gdn_oracle_kda_replay(K, V, ntok[i], S, rec_u + rec * V, rec_k + rec * K,
                            rec_g + rec * K);
      memcpy(pools_out + l * pool_elems + ((size_t)slots[i] * HV + h) * VK, S,
             VK * sizeof(double));
    }
    free(S);
  }
  return 0;
}
