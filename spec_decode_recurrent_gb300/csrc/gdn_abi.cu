// gdn_abi.cu -- the extern "C" entry points of libgdn_spec.so: host-side
// validation, then one kernel launch each.  See include/gdn_spec.h for the
// contract of every argument.
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_launch.h"
#include "gdn_spec.h"

namespace {

bool supported_width(int x) { return x == 16 || x == 32 || x == 64 || x == 128; }
bool aligned(const void* ptr, uintptr_t bytes) {
  return (reinterpret_cast<uintptr_t>(ptr) & (bytes - 1)) == 0;
}
bool valid_dtype(int d) { return d == GDN_DTYPE_F32 || d == GDN_DTYPE_BF16; }
size_t dtype_bytes(int d) { return d == GDN_DTYPE_BF16 ? 2 : 4; }

int check_shape(const gdn_shape* s) {
  if (!s) return GDN_ERR_NULL;
  if (s->num_k_heads < 1 || s->num_v_heads < 1 || s->num_v_heads % s->num_k_heads != 0 ||
      s->num_v_heads > 65535)
    return GDN_ERR_UNSUPPORTED;
  if (!supported_width(s->head_k) || !supported_width(s->head_v)) return GDN_ERR_UNSUPPORTED;
  if (s->max_window < 1 || s->max_window > gdn::kMaxWindow) return GDN_ERR_UNSUPPORTED;
  if (!valid_dtype(s->qkv_dtype) || !valid_dtype(s->state_dtype)) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

// Checks shared by the verify and the native snapshot, and the parameter block.
int prepare_verify(gdn::VerifyParams* p, const gdn_shape* s, int32_t batch,
                   int32_t num_tokens, int32_t num_slots, const void* q,
                   int64_t q_row_stride, const void* k, int64_t k_row_stride,
                   const void* v, int64_t v_row_stride, const float* a,
                   const float* b, const float* A_log, const float* dt_bias,
                   const int32_t* token_start, const int32_t* window_len,
                   const void* state_pool, const int32_t* slot_table,
                   int32_t slot_table_stride, const int32_t* seq_pos,
                   int32_t block_size, float* out, int64_t out_row_stride) {
  int rc = check_shape(s);
  if (rc != GDN_OK) return rc;
  if (!q || !k || !v || !a || !b || !A_log || !dt_bias || !token_start || !window_len ||
      !state_pool || !slot_table || !out)
    return GDN_ERR_NULL;
  if (block_size < 0 || slot_table_stride < 1) return GDN_ERR_INVALID;
  if (block_size > 0 && !seq_pos) return GDN_ERR_NULL;
  if (batch < 0 || batch > 65535 || num_tokens < 0 || num_slots < 0) return GDN_ERR_INVALID;
  const int64_t qk_row = (int64_t)s->num_k_heads * s->head_k;
  const int64_t v_row = (int64_t)s->num_v_heads * s->head_v;
  if (q_row_stride < qk_row || k_row_stride < qk_row || v_row_stride < v_row ||
      out_row_stride < v_row)
    return GDN_ERR_INVALID;
  if (q_row_stride % 4 || k_row_stride % 4) return GDN_ERR_INVALID;
  const uintptr_t qk_align = 4 * dtype_bytes(s->qkv_dtype);
  if (!aligned(q, qk_align) || !aligned(k, qk_align) || !aligned(v, dtype_bytes(s->qkv_dtype)))
    return GDN_ERR_INVALID;
  if (!aligned(state_pool, 16) || !aligned(out, 4) || !aligned(a, 4) || !aligned(b, 4))
    return GDN_ERR_INVALID;

  p->HK = s->num_k_heads;
  p->HV = s->num_v_heads;
  p->V = s->head_v;
  p->W = s->max_window;
  p->batch = batch;
  p->num_tokens = num_tokens;
  p->num_slots = num_slots;
  p->q = q;
  p->k = k;
  p->v = v;
  p->q_stride = q_row_stride;
  p->k_stride = k_row_stride;
  p->v_stride = v_row_stride;
  p->a = a;
  p->b = b;
  p->A_log = A_log;
  p->dt_bias = dt_bias;
  p->token_start = token_start;
  p->window_len = window_len;
  p->pool = state_pool;
  p->slot_table = slot_table;
  p->table_stride = slot_table_stride;
  p->seq_pos = seq_pos;
  p->block_size = block_size;
  p->out = out;
  p->out_stride = out_row_stride;
  p->rec_u = nullptr;
  p->rec_k = nullptr;
  p->rec_g = nullptr;
  p->snaps = nullptr;
  p->err = nullptr;
  return GDN_OK;
}

int verify_common(const gdn_shape* shape, int32_t batch, int32_t num_tokens, int32_t num_slots,
                  const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                  const void* v, int64_t v_row_stride, const float* a, const float* b,
                  const float* A_log, const float* dt_bias, const int32_t* token_start,
                  const int32_t* window_len, const void* state_pool, const int32_t* slot_table,
                  int32_t slot_table_stride, const int32_t* seq_pos, int32_t block_size,
                  float* out, int64_t out_row_stride, float* rec_u, float* rec_k, float* rec_g,
                  void* snapshots, int32_t* err, void* stream, bool native, bool kda) {
  if (batch == 0) return check_shape(shape);  // nothing to do; row arrays may be empty
  gdn::VerifyParams p;
  int rc = prepare_verify(&p, shape, batch, num_tokens, num_slots, q, q_row_stride, k,
                          k_row_stride, v, v_row_stride, a, b, A_log, dt_bias, token_start,
                          window_len, state_pool, slot_table, slot_table_stride, seq_pos,
                          block_size, out, out_row_stride);
  if (rc != GDN_OK) return rc;
  if (native) {
    if (!snapshots) return GDN_ERR_NULL;
    if (!aligned(snapshots, 16)) return GDN_ERR_INVALID;
    p.snaps = snapshots;
  } else {
    if (!rec_u || !rec_k || !rec_g) return GDN_ERR_NULL;
    // a per-channel gate record moves in 16-byte pieces
    if (!aligned(rec_u, 16) || !aligned(rec_k, 16) || !aligned(rec_g, kda ? 16 : 4))
      return GDN_ERR_INVALID;
    p.rec_u = rec_u;
    p.rec_k = rec_k;
    p.rec_g = rec_g;
  }
  p.err = err;
  return gdn::launch_verify(p, shape->head_k, shape->qkv_dtype, shape->state_dtype, native, kda,
                            static_cast<cudaStream_t>(stream));
}

int commit_common(const gdn_shape* shape, int32_t num_layers, int32_t num_groups,
                  const int32_t* layer_group, int32_t batch, int32_t num_slots,
                  void* const* state_pools, const float* const* rec_u, const float* const* rec_k,
                  const float* const* rec_g, const int32_t* window_len,
                  const int32_t* accepted_len, const int32_t* slot_tables,
                  int32_t slot_table_stride, int64_t group_stride, const int32_t* seq_pos,
                  int32_t block_size, int32_t* err, void* stream, bool kda) {
  int rc = check_shape(shape);
  if (rc != GDN_OK || batch == 0) return rc;
  if (!state_pools || !rec_u || !rec_k || !rec_g || !window_len || !accepted_len ||
      !slot_tables)
    return GDN_ERR_NULL;
  if (num_groups > 1 && !layer_group) return GDN_ERR_NULL;
  if (block_size < 0 || slot_table_stride < 1) return GDN_ERR_INVALID;
  if (block_size > 0 && !seq_pos) return GDN_ERR_NULL;
  if (num_layers < 1 || num_layers > 65535 || batch < 0 || batch > 65535 || num_slots < 0 ||
      num_groups < 1)
    return GDN_ERR_INVALID;
  if (num_groups > 1 && group_stride < (int64_t)batch * slot_table_stride) return GDN_ERR_INVALID;
  gdn::CommitParams p;
  p.HV = shape->num_v_heads;
  p.V = shape->head_v;
  p.W = shape->max_window;
  p.num_layers = num_layers;
  p.batch = batch;
  p.num_slots = num_slots;
  p.layer_group = layer_group;
  p.num_groups = num_groups;
  p.group_stride = num_groups > 1 ? group_stride : 0;
  p.pools = state_pools;
  p.rec_u = rec_u;
  p.rec_k = rec_k;
  p.rec_g = rec_g;
  p.window_len = window_len;
  p.accepted_len = accepted_len;
  p.slot_table = slot_tables;
  p.table_stride = slot_table_stride;
  p.seq_pos = seq_pos;
  p.block_size = block_size;
  p.err = err;
  return gdn::launch_commit(p, shape->head_k, shape->state_dtype, kda,
                            static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

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
                    void* stream) {
  return verify_common(shape, batch, num_tokens, num_slots, q, q_row_stride, k, k_row_stride, v,
                       v_row_stride, a, b, A_log, dt_bias, token_start, window_len, state_pool,
                       slot_table, slot_table_stride, seq_pos, block_size, out, out_row_stride,
                       rec_u, rec_k, rec_g, nullptr, err, stream, false, false);
}

int gdn_native_spec_snapshot(
    const gdn_shape* shape, int32_t batch, int32_t num_tokens, int32_t num_slots,
    const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
    int64_t v_row_stride, const float* a, const float* b, const float* A_log,
    const float* dt_bias, const int32_t* token_start, const int32_t* window_len,
    const void* state_pool, const int32_t* slot_table, int32_t slot_table_stride,
    const int32_t* seq_pos, int32_t block_size, float* out, int64_t out_row_stride,
    void* snapshots, int32_t* err, void* stream) {
  return verify_common(shape, batch, num_tokens, num_slots, q, q_row_stride, k, k_row_stride, v,
                       v_row_stride, a, b, A_log, dt_bias, token_start, window_len, state_pool,
                       slot_table, slot_table_stride, seq_pos, block_size, out, out_row_stride,
                       nullptr, nullptr, nullptr, snapshots, err, stream, true, false);
}

int gdn_kda_spec_verify(const gdn_shape* shape, int32_t batch, int32_t num_tokens,
                        int32_t num_slots, const void* q, int64_t q_row_stride, const void* k,
                        int64_t k_row_stride, const void* v, int64_t v_row_stride,
                        const float* a, const float* b, const float* A_log,
                        const float* dt_bias, const int32_t* token_start,
                        const int32_t* window_len, const void* state_pool,
                        const int32_t* slot_table, int32_t slot_table_stride,
                        const int32_t* seq_pos, int32_t block_size, float* out,
                        int64_t out_row_stride, float* rec_u, float* rec_k, float* rec_g,
                        int32_t* err, void* stream) {
  return verify_common(shape, batch, num_tokens, num_slots, q, q_row_stride, k, k_row_stride, v,
                       v_row_stride, a, b, A_log, dt_bias, token_start, window_len, state_pool,
                       slot_table, slot_table_stride, seq_pos, block_size, out, out_row_stride,
                       rec_u, rec_k, rec_g, nullptr, err, stream, false, true);
}

int gdn_kda_native_spec_snapshot(
    const gdn_shape* shape, int32_t batch, int32_t num_tokens, int32_t num_slots,
    const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
    int64_t v_row_stride, const float* a, const float* b, const float* A_log,
    const float* dt_bias, const int32_t* token_start, const int32_t* window_len,
    const void* state_pool, const int32_t* slot_table, int32_t slot_table_stride,
    const int32_t* seq_pos, int32_t block_size, float* out, int64_t out_row_stride,
    void* snapshots, int32_t* err, void* stream) {
  return verify_common(shape, batch, num_tokens, num_slots, q, q_row_stride, k, k_row_stride, v,
                       v_row_stride, a, b, A_log, dt_bias, token_start, window_len, state_pool,
                       slot_table, slot_table_stride, seq_pos, block_size, out, out_row_stride,
                       nullptr, nullptr, nullptr, snapshots, err, stream, true, true);
}

int gdn_replay_commit_grouped(const gdn_shape* shape, int32_t num_layers, int32_t num_groups,
                              const int32_t* layer_group, int32_t batch, int32_t num_slots,
                              void* const* state_pools, const float* const* rec_u,
                              const float* const* rec_k, const float* const* rec_g,
                              const int32_t* window_len, const int32_t* accepted_len,
                              const int32_t* slot_tables, int32_t slot_table_stride,
                              int64_t group_stride, const int32_t* seq_pos, int32_t block_size,
                              int32_t* err, void* stream) {
  return commit_common(shape, num_layers, num_groups, layer_group, batch, num_slots, state_pools,
                       rec_u, rec_k, rec_g, window_len, accepted_len, slot_tables,
                       slot_table_stride, group_stride, seq_pos, block_size, err, stream, false);
}

int gdn_replay_commit(const gdn_shape* shape, int32_t num_layers, int32_t batch,
                      int32_t num_slots, void* const* state_pools, const float* const* rec_u,
                      const float* const* rec_k, const float* const* rec_g,
                      const int32_t* window_len, const int32_t* accepted_len,
                      const int32_t* slot_table, int32_t slot_table_stride,
                      const int32_t* seq_pos, int32_t block_size, int32_t* err,
                      void* stream) {
  return commit_common(shape, num_layers, 1, nullptr, batch, num_slots, state_pools, rec_u,
                       rec_k, rec_g, window_len, accepted_len, slot_table, slot_table_stride, 0,
                       seq_pos, block_size, err, stream, false);
}

int gdn_kda_replay_commit_grouped(const gdn_shape* shape, int32_t num_layers,
                                  int32_t num_groups, const int32_t* layer_group, int32_t batch,
                                  int32_t num_slots, void* const* state_pools,
                                  const float* const* rec_u, const float* const* rec_k,
                                  const float* const* rec_g, const int32_t* window_len,
                                  const int32_t* accepted_len, const int32_t* slot_tables,
                                  int32_t slot_table_stride, int64_t group_stride,
                                  const int32_t* seq_pos, int32_t block_size, int32_t* err,
                                  void* stream) {
  return commit_common(shape, num_layers, num_groups, layer_group, batch, num_slots, state_pools,
                       rec_u, rec_k, rec_g, window_len, accepted_len, slot_tables,
                       slot_table_stride, group_stride, seq_pos, block_size, err, stream, true);
}

int gdn_kda_replay_commit(const gdn_shape* shape, int32_t num_layers, int32_t batch,
                          int32_t num_slots, void* const* state_pools,
                          const float* const* rec_u, const float* const* rec_k,
                          const float* const* rec_g, const int32_t* window_len,
                          const int32_t* accepted_len, const int32_t* slot_table,
                          int32_t slot_table_stride, const int32_t* seq_pos, int32_t block_size,
                          int32_t* err, void* stream) {
  return commit_common(shape, num_layers, 1, nullptr, batch, num_slots, state_pools, rec_u,
                       rec_k, rec_g, window_len, accepted_len, slot_table, slot_table_stride, 0,
                       seq_pos, block_size, err, stream, true);
}

int gdn_conv_state_commit(int32_t num_layers, int32_t num_groups, const int32_t* layer_group,
                          int32_t batch, int32_t num_tokens, int32_t num_slots, int32_t channels,
                          int32_t state_len, int32_t dtype, int32_t max_window,
                          void* const* conv_pools, const void* const* conv_inputs,
                          int64_t input_row_stride, const int32_t* token_start,
                          const int32_t* window_len, const int32_t* accepted_len,
                          const int32_t* slot_tables, int32_t slot_table_stride,
                          int64_t group_stride, const int32_t* seq_pos, int32_t block_size,
                          int32_t* err, void* stream) {
  if (channels < 1 || state_len < 1 || state_len > 8 || !valid_dtype(dtype) || max_window < 1 ||
      max_window > gdn::kMaxWindow)
    return GDN_ERR_UNSUPPORTED;
  if (batch == 0) return GDN_OK;
  if (!conv_pools || !conv_inputs || !token_start || !window_len || !accepted_len || !slot_tables)
    return GDN_ERR_NULL;
  if (num_groups > 1 && !layer_group) return GDN_ERR_NULL;
  if (block_size > 0 && !seq_pos) return GDN_ERR_NULL;
  if (num_layers < 1 || num_layers > 65535 || batch < 0 || batch > 65535 || num_slots < 0 ||
      num_tokens < 0 || num_groups < 1 || block_size < 0 || slot_table_stride < 1 ||
      input_row_stride < channels || channels % 8 != 0 || input_row_stride % 8 != 0)
    return GDN_ERR_INVALID;
  if (num_groups > 1 && group_stride < (int64_t)batch * slot_table_stride) return GDN_ERR_INVALID;
  gdn::ConvParams p;
  p.num_layers = num_layers;
  p.batch = batch;
  p.num_slots = num_slots;
  p.num_tokens = num_tokens;
  p.C = channels;
  p.SL = state_len;
  p.W = max_window;
  p.layer_group = layer_group;
  p.num_groups = num_groups;
  p.group_stride = num_groups > 1 ? group_stride : 0;
  p.pools = conv_pools;
  p.inputs = conv_inputs;
  p.in_stride = input_row_stride;
  p.token_start = token_start;
  p.window_len = window_len;
  p.accepted_len = accepted_len;
  p.slot_table = slot_tables;
  p.table_stride = slot_table_stride;
  p.seq_pos = seq_pos;
  p.block_size = block_size;
  p.err = err;
  return gdn::launch_conv_commit(p, dtype, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
