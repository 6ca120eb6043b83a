/*
 * gdn_spec.h -- C ABI of libgdn_spec.so: speculative (MTP) verify and
 * all-layer replay commit for Gated DeltaNet (GDN) layers on one GPU.
 *
 * The method (vLLM PR "[Spec Decode][Qwen4Exp] RecoverSSM for Qwen GDN and
 * the PLE short conv", Purpose; tokenspeed PR "feat: add Qwen3.5 GDN
 * ReplaySSM", Summary and Motivation):
 *   - the verify runs each request's draft window from a read-only
 *     checkpoint state, writes the per-token outputs and a small per-token
 *     replay record [correction u (V), normalized key (K), gate (1)] in
 *     fp32, and writes no state;
 *   - after sampling, one commit launch over all layers replays only the
 *     accepted prefix, h = fma(u, k, h * decay), and writes each state once
 *     (plus the block-boundary state in align mode);
 *   - the native baseline instead stores the full state after every draft
 *     position.
 *
 * Recurrence, per value head h with a [V][K] fp32 state S (K contiguous):
 *   alpha_t = exp(-exp(A_log[h]) * softplus(a[t,h] + dt_bias[h]))
 *   beta_t  = sigmoid(b[t,h])
 *   khat_t  = k_t / sqrt(|k_t|^2 + 1e-6),  qhat_t likewise
 *   H = alpha_t * S;  u_t = beta_t * (v_t - H khat_t);  S = H + u_t khat_t^T
 *   o_t = S qhat_t
 * Value head h reads key head h / (num_v_heads / num_k_heads).
 * All three kernels run the same fp32 operations in the same order, so the
 * verify's outputs equal the native kernel's and a commit after n accepted
 * tokens equals the native state after token n, bit for bit.
 *
 * Conventions for every entry point:
 *   - Every pointer is device memory owned by the caller, except `shape`,
 *     which is a host pointer read during the call only.  The library never
 *     allocates, frees or synchronises; it enqueues kernels on `stream`
 *     (a cudaStream_t; NULL = legacy default stream) on the current device
 *     and returns.
 *   - Return value: GDN_OK, or a negative GDN_ERR_* for a problem the host
 *     can see (null pointer, unsupported shape, bad stride or alignment,
 *     failed launch).  Nothing is launched when the return is negative.
 *     batch == 0 launches nothing and checks only the shape (the per-row
 *     arrays of an empty batch may be NULL).
 *   - Row-level problems are found on the device: the row is skipped and
 *     its GDN_ROW_ERR_* bits are OR-ed into *err when err is not NULL.  The
 *     caller clears *err beforehand.  A skipped row writes nothing, with one
 *     exception: gdn_spec_verify marks a row it rejects by writing -1.0 (a
 *     value no decay takes) into rec_g[r][h][0] for every head h, and
 *     gdn_replay_commit stores nothing for a row whose record carries that
 *     marker (GDN_ROW_ERR_REJECTED), so a verify-rejected row is never
 *     committed even when no host code reads *err in between.
 *   - Null rows: a row whose window_len is 0 or whose checkpoint slot is -1
 *     reads and writes nothing (graph padding rows; vLLM PR above, Purpose).
 *   - Slot of the state after x folded tokens of row r:
 *       block_size == 0: slot_table[r * slot_table_stride + 0]
 *       block_size  > 0: slot_table[r * slot_table_stride + (x - 1) / block_size]
 *     (align mode: a state lives in the block of its last token; vLLM PR
 *     above, Commits item 3).  The checkpoint is the state after
 *     x = seq_pos[r] tokens; seq_pos is read only in align mode.
 *
 * Supported shapes: head_k, head_v in {16, 32, 64, 128}; max_window 1..16;
 * num_v_heads a multiple of num_k_heads and <= 65535; batch, num_layers <=
 * 65535.
 */
#ifndef GDN_SPEC_H_
#define GDN_SPEC_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
#define GDN_DTYPE_F32 0
#define GDN_DTYPE_BF16 1

/* Return codes. */
#define GDN_OK 0
#define GDN_ERR_NULL (-1)        /* a required pointer is NULL                */
#define GDN_ERR_UNSUPPORTED (-2) /* shape or dtype outside the supported set  */
#define GDN_ERR_INVALID (-3)     /* bad count, stride, alignment or block size */
#define GDN_ERR_CUDA (-4)        /* the kernel launch failed                   */

/* Row error bits OR-ed into *err. */
#define GDN_ROW_ERR_WINDOW 1     /* window_len outside [0, max_window]                */
#define GDN_ROW_ERR_ACCEPTED 2   /* accepted_len outside [0, window_len]              */
#define GDN_ROW_ERR_SLOT 4       /* slot outside [-1, num_slots)                      */
#define GDN_ROW_ERR_BLOCK 8      /* align mode: a needed column is outside the table, */
                                 /* or holds -1 although the row is live             */
#define GDN_ROW_ERR_SEQPOS 16    /* align mode: seq_pos < 1 on a live row             */
#define GDN_ROW_ERR_TOKENS 32    /* token rows outside [0, num_tokens)                */
#define GDN_ROW_ERR_GROUP 64     /* grouped commit: a layer's group id is outside     */
                                 /* [0, num_groups); that layer writes nothing       */
#define GDN_ROW_ERR_REJECTED 128 /* commit: the verify rejected this row (its gate    */
                                 /* record holds the reject marker); nothing stored  */
#define GDN_ROW_ERR_TIMEOUT 256  /* a CTA gave up waiting for its own asynchronous    */
                                 /* copy (never expected); its remaining work is not */
                                 /* done and the call's outputs are incomplete       */

typedef struct gdn_shape {
  int32_t num_k_heads; /* HK                                              */
  int32_t num_v_heads; /* HV, a multiple of HK                            */
  int32_t head_k;      /* K: key width, the state's contiguous dimension   */
  int32_t head_v;      /* V: value width, the state's row count            */
  int32_t max_window;  /* W: record stride in tokens, 1..16                */
  int32_t qkv_dtype;   /* GDN_DTYPE_F32 or GDN_DTYPE_BF16 for q, k, v      */
  int32_t state_dtype; /* GDN_DTYPE_F32 or GDN_DTYPE_BF16 for the state    */
} gdn_shape;

/*
 * Speculative verify of one layer (vLLM PR above, Purpose and Commits
 * item 2: the verify reads strided q/k/v views of the conv output and
 * writes straight into the layer output).
 *
 *   q, k          [num_tokens][HK][K] of qkv_dtype; token row t starts at
 *                 q + t * q_row_stride (elements), heads contiguous inside a
 *                 row.  Base 16-byte aligned (fp32) or 8-byte (bf16); row
 *                 stride a multiple of 4 elements.
 *   v             [num_tokens][HV][V] of qkv_dtype, row stride v_row_stride.
 *   a, b          [num_tokens][HV] fp32, contiguous: raw gate inputs.
 *   A_log, dt_bias [HV] fp32.
 *   token_start, window_len [batch] int32: row r owns token rows
 *                 token_start[r] .. token_start[r] + window_len[r] - 1.
 *                 Rows need not be contiguous or ordered.
 *   state_pool    [num_slots][HV][V][K] of state_dtype, 16-byte aligned.
 *                 Read only: the checkpoint is never written.
 *   slot_table    [batch][slot_table_stride] int32; seq_pos [batch] int32
 *                 (align mode only, else may be NULL); block_size >= 0.
 *   out           [num_tokens][HV][V] fp32, row stride out_row_stride:
 *                 o_t for every token of every live row; other rows are not
 *                 touched.
 *   rec_u [batch][HV][W][V], rec_k [batch][HV][W][K], rec_g [batch][HV][W]
 *                 fp32, 16-byte aligned: the replay record of token t of row
 *                 r in position t; positions >= window_len[r] are untouched.
 *   err           optional int32 row-error word.
 */
int gdn_spec_verify(const gdn_shape* shape, int32_t batch, int32_t num_tokens,
                    int32_t num_slots, const void* q, int64_t q_row_stride,
                    const void* k, int64_t k_row_stride, const void* v,
                    int64_t v_row_stride, const float* a, const float* b,
                    const float* A_log, const float* dt_bias,
                    const int32_t* token_start, const int32_t* window_len,
                    const void* state_pool, const int32_t* slot_table,
                    int32_t slot_table_stride, const int32_t* seq_pos,
                    int32_t block_size, float* out, int64_t out_row_stride,
                    float* rec_u, float* rec_k, float* rec_g, int32_t* err,
                    void* stream);

/*
 * All-layer replay commit in one launch (tokenspeed PR above, Summary and
 * Implementation: layer-indexed state pools and replay buffers, a single
 * replay kernel over all GDN layers; vLLM PR above, Purpose and Commits
 * items 3 and 6).
 *
 *   state_pools   device array of num_layers device pointers, each to a
 *                 [num_slots][HV][V][K] pool of state_dtype (16-byte
 *                 aligned), updated in place.
 *   rec_u, rec_k, rec_g  device arrays of num_layers device pointers to the
 *                 layer's records, laid out as gdn_spec_verify writes them.
 *   window_len, accepted_len [batch] int32; slot_table, seq_pos, block_size
 *                 as for gdn_spec_verify (the same values the verify saw).
 * For each live row with n = accepted_len[r] > 0 the state after n tokens
 * is written to slot(seq_pos + n) (slot(n) without align mode, i.e. in
 * place).  In align mode each block boundary p with seq_pos < p <
 * seq_pos + n, p % block_size == 0, also receives the state after
 * p - seq_pos tokens in slot(p); a boundary at seq_pos + n is the final
 * state and is written once.  Every write starts from the unmodified
 * checkpoint, so a boundary slot equal to the checkpoint slot is safe
 * (final folds before boundary folds).  A bf16 state is rounded once per
 * stored state (round to nearest even).  Rows with n == 0 or a null slot
 * write nothing; a row whose gate record holds the verify's reject marker
 * writes nothing and sets GDN_ROW_ERR_REJECTED.
 *
 * Slots are not shared between rows: every slot a live row writes (its final
 * and boundary slots) must be neither read nor written by any other live
 * row of the same call, in any layer group.  Rows run concurrently with no
 * ordering between them, so a shared slot gives a timing-dependent result.
 * Within one row, a boundary or final slot equal to its own checkpoint slot
 * is fine (see above).
 */
int gdn_replay_commit(const gdn_shape* shape, int32_t num_layers,
                      int32_t batch, int32_t num_slots,
                      void* const* state_pools, const float* const* rec_u,
                      const float* const* rec_k, const float* const* rec_g,
                      const int32_t* window_len, const int32_t* accepted_len,
                      const int32_t* slot_table, int32_t slot_table_stride,
                      const int32_t* seq_pos, int32_t block_size, int32_t* err,
                      void* stream);

/*
 * Grouped all-layer commit: one launch covering every KV-cache group, for
 * engines whose GDN layers are split into groups with their own state
 * indices (vLLM PR above, review thread: a grouped commit over a
 * [group, batch] state-index table instead of one commit per group).
 *
 *   num_groups     >= 1
 *   layer_group    device int32 [num_layers]: group of each layer.
 *   slot_tables    device int32 [num_groups][batch][slot_table_stride];
 *                  group g's table starts group_stride elements after
 *                  group g-1's (group_stride >= batch * slot_table_stride).
 * Everything else as gdn_replay_commit, whose semantics each layer follows
 * with its group's table.  Row errors are OR-ed over all groups; a layer
 * with an out-of-range group id writes nothing and sets GDN_ROW_ERR_GROUP.
 */
int gdn_replay_commit_grouped(const gdn_shape* shape, int32_t num_layers,
                              int32_t num_groups, const int32_t* layer_group,
                              int32_t batch, int32_t num_slots,
                              void* const* state_pools,
                              const float* const* rec_u,
                              const float* const* rec_k,
                              const float* const* rec_g,
                              const int32_t* window_len,
                              const int32_t* accepted_len,
                              const int32_t* slot_tables,
                              int32_t slot_table_stride, int64_t group_stride,
                              const int32_t* seq_pos, int32_t block_size,
                              int32_t* err, void* stream);

/*
 * Short-conv state commit over all layers in one launch (vLLM PR above,
 * Purpose: the short-conv state is advanced over the accepted tokens by the
 * recurrent commit's own plan; Commits item 1: the commit's plan, conv and
 * state steps).  A layer's
 * causal depthwise convolution of width state_len + 1 keeps, per slot and
 * channel, the last state_len convolution inputs, oldest first.  For each
 * live row with n = accepted_len[r] > 0 the state after x tokens -- the last
 * state_len entries of (checkpoint state ++ the row's first x inputs) -- is
 * written to the slots gdn_replay_commit writes for x = n (and, in align
 * mode, for each boundary).  Pure copies: results are bit-exact.
 *
 *   channels, state_len  C a multiple of 8, 1 <= state_len <= 8; dtype:
 *                  element type of both the state and the inputs (F32 or
 *                  BF16).
 *   conv_pools     device array [num_layers] of device pointers to
 *                  [num_slots][C][state_len] states, 16-byte aligned,
 *                  updated in place.
 *   conv_inputs    device array [num_layers] of device pointers to the
 *                  layer's convolution inputs, one row of C elements per
 *                  token row, rows input_row_stride elements apart (a
 *                  multiple of 8); each pointer 16-byte aligned.
 *   token_start    [batch]: first token row of each request's window.
 *   layer_group / num_groups / slot_tables / group_stride as in
 *                  gdn_replay_commit_grouped (num_groups = 1 and layer_group
 *                  NULL for a single table).
 * Row errors as for the commit, plus GDN_ROW_ERR_TOKENS for window rows
 * outside [0, num_tokens).
 */
int gdn_conv_state_commit(int32_t num_layers, int32_t num_groups,
                          const int32_t* layer_group, int32_t batch,
                          int32_t num_tokens, int32_t num_slots,
                          int32_t channels, int32_t state_len, int32_t dtype,
                          int32_t max_window, void* const* conv_pools,
                          const void* const* conv_inputs,
                          int64_t input_row_stride, const int32_t* token_start,
                          const int32_t* window_len,
                          const int32_t* accepted_len,
                          const int32_t* slot_tables,
                          int32_t slot_table_stride, int64_t group_stride,
                          const int32_t* seq_pos, int32_t block_size,
                          int32_t* err, void* stream);

/*
 * Native baseline of one layer: the verify's recurrence with the full
 * state stored after every draft position, and no record (vLLM PR above,
 * Purpose: the path that snapshots the recurrent state after every draft
 * position; tokenspeed PR above, Motivation).
 *
 * Arguments as gdn_spec_verify up to out_row_stride, then
 *   snapshots     [batch][W][HV][V][K] of state_dtype, 16-byte aligned:
 *                 snapshots[r][t] = state after token t of row r
 *                 (t < window_len[r]); a bf16 state is rounded once per
 *                 stored snapshot.  Other positions are untouched and the
 *                 checkpoint pool is never written.
 */
int gdn_native_spec_snapshot(
    const gdn_shape* shape, int32_t batch, int32_t num_tokens,
    int32_t num_slots, const void* q, int64_t q_row_stride, const void* k,
    int64_t k_row_stride, const void* v, int64_t v_row_stride, const float* a,
    const float* b, const float* A_log, const float* dt_bias,
    const int32_t* token_start, const int32_t* window_len,
    const void* state_pool, const int32_t* slot_table,
    int32_t slot_table_stride, const int32_t* seq_pos, int32_t block_size,
    float* out, int64_t out_row_stride, void* snapshots, int32_t* err,
    void* stream);

/*
 * Per-channel decay (KDA) variant of the three calls above.  The pages
 * name KDA as the layer the verify/commit protocol was first built for
 * (tokenspeed PR above, Summary; vLLM PR above, Purpose) but print no KDA
 * formula; the reading implemented here replaces the scalar decay by a
 * vector over the K key channels and changes nothing else:
 *   alpha_t[j] = exp(-exp(A_log[h]) * softplus(a[t,h,j] + dt_bias[h,j]))
 *   H = S diag(alpha_t)   (column j of the [V][K] state scaled by alpha_t[j])
 *   u_t = beta_t * (v_t - H khat_t);  S = H + u_t khat_t^T;  o_t = S qhat_t
 * and the replay record keeps the whole gate vector.  The commit's fold is
 * S[i][j] = fma(u[i], khat[j], S[i][j] * alpha[j]), so, as for the scalar
 * gate, verify == native and commit(n) == native snapshot n bit for bit.
 *
 * Arguments exactly as gdn_spec_verify / gdn_native_spec_snapshot /
 * gdn_replay_commit, except these layouts:
 *   a             [num_tokens][HV][K] fp32, contiguous: per-channel raw gates.
 *   dt_bias       [HV][K] fp32.
 *   rec_g         [batch][HV][W][K] fp32, 16-byte aligned (verify output,
 *                 commit input through its pointer array): the gate vector
 *                 of token t of row r in position t.  The reject marker is
 *                 rec_g[r][h][0][0] = -1.0.
 */
int gdn_kda_spec_verify(const gdn_shape* shape, int32_t batch, int32_t num_tokens,
                        int32_t num_slots, const void* q, int64_t q_row_stride,
                        const void* k, int64_t k_row_stride, const void* v,
                        int64_t v_row_stride, const float* a, const float* b,
                        const float* A_log, const float* dt_bias,
                        const int32_t* token_start, const int32_t* window_len,
                        const void* state_pool, const int32_t* slot_table,
                        int32_t slot_table_stride, const int32_t* seq_pos,
                        int32_t block_size, float* out, int64_t out_row_stride,
                        float* rec_u, float* rec_k, float* rec_g, int32_t* err,
                        void* stream);

int gdn_kda_native_spec_snapshot(
    const gdn_shape* shape, int32_t batch, int32_t num_tokens,
    int32_t num_slots, const void* q, int64_t q_row_stride, const void* k,
    int64_t k_row_stride, const void* v, int64_t v_row_stride, const float* a,
    const float* b, const float* A_log, const float* dt_bias,
    const int32_t* token_start, const int32_t* window_len,
    const void* state_pool, const int32_t* slot_table,
    int32_t slot_table_stride, const int32_t* seq_pos, int32_t block_size,
    float* out, int64_t out_row_stride, void* snapshots, int32_t* err,
    void* stream);

int gdn_kda_replay_commit(const gdn_shape* shape, int32_t num_layers,
                          int32_t batch, int32_t num_slots,
                          void* const* state_pools, const float* const* rec_u,
                          const float* const* rec_k, const float* const* rec_g,
                          const int32_t* window_len,
                          const int32_t* accepted_len,
                          const int32_t* slot_table, int32_t slot_table_stride,
                          const int32_t* seq_pos, int32_t block_size,
                          int32_t* err, void* stream);

/* The grouped all-layer commit (arguments as gdn_replay_commit_grouped) with
 * per-channel gate records [batch][HV][W][K]. */
int gdn_kda_replay_commit_grouped(const gdn_shape* shape, int32_t num_layers,
                                  int32_t num_groups, const int32_t* layer_group,
                                  int32_t batch, int32_t num_slots,
                                  void* const* state_pools,
                                  const float* const* rec_u,
                                  const float* const* rec_k,
                                  const float* const* rec_g,
                                  const int32_t* window_len,
                                  const int32_t* accepted_len,
                                  const int32_t* slot_tables,
                                  int32_t slot_table_stride, int64_t group_stride,
                                  const int32_t* seq_pos, int32_t block_size,
                                  int32_t* err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_SPEC_H_ */
