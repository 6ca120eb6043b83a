// gdn_device.cuh -- device helpers shared by the verify, native-snapshot and
// commit kernels of libgdn_spec.so.
//
// Every floating-point step of the recurrence is written with explicit
// round-to-nearest intrinsics (__fmul_rn, __fmaf_rn, ...) and the library is
// compiled with -fmad=false, so no kernel can contract a multiply and an add
// differently from another.  That is what makes the verify's outputs equal
// to the native kernel's, and a commit after n accepted tokens equal to the
// native state after token n, bit for bit (vLLM PR "[Spec Decode][Qwen4Exp]
// RecoverSSM for Qwen GDN and the PLE short conv", Test Result: the commit
// replays forward with the same update h = fma(c, k, h * decay)).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "gdn_spec.h"

namespace gdn {

constexpr int kMaxWindow = 16;
constexpr float kL2NormEps = 1e-6f;
// Written by the verify into gate record position 0 of every head of a row
// it rejects; no decay exp(g) is negative, so the commit recognises it and
// skips the row without storing anything.
constexpr float kRejectedGate = -1.0f;

// ------------------------------------------------------------ parameters
struct VerifyParams {
  int HK, HV, V, W;
  int batch, num_tokens, num_slots;
  const void* q;
  const void* k;
  const void* v;
  long long q_stride, k_stride, v_stride;  // elements per token row
  const float* a;
  const float* b;
  const float* A_log;
  const float* dt_bias;
  const int32_t* token_start;
  const int32_t* window_len;
  const void* pool;
  const int32_t* slot_table;
  int table_stride;
  const int32_t* seq_pos;
  int block_size;
  float* out;
  long long out_stride;
  float* rec_u;
  float* rec_k;
  float* rec_g;
  void* snaps;
  int32_t* err;
};

struct CommitParams {
  int HV, V, W;
  int num_layers, batch, num_slots;
  const int32_t* layer_group;  // [num_layers] or NULL (one group)
  int num_groups;
  long long group_stride;      // elements between two groups' slot tables
  void* const* pools;
  const float* const* rec_u;
  const float* const* rec_k;
  const float* const* rec_g;
  const int32_t* window_len;
  const int32_t* accepted_len;
  const int32_t* slot_table;
  int table_stride;
  const int32_t* seq_pos;
  int block_size;
  int32_t* err;
};

struct ConvParams {
  int num_layers, batch, num_slots, num_tokens;
  int C, SL, W;                  // channels, state length, max window
  const int32_t* layer_group;    // [num_layers] or NULL (one group)
  int num_groups;
  long long group_stride;
  void* const* pools;            // [num_layers] -> [num_slots][C][SL]
  const void* const* inputs;     // [num_layers] -> token rows of C inputs
  long long in_stride;           // elements between token rows
  const int32_t* token_start;
  const int32_t* window_len;
  const int32_t* accepted_len;
  const int32_t* slot_table;
  int table_stride;
  const int32_t* seq_pos;
  int block_size;
  int32_t* err;
};

// ----------------------------------------------------------------- gates
// softplus(x) = log(1 + e^x), in the form that does not overflow.
__device__ __forceinline__ float softplus(float x) {
  return x > 0.0f ? __fadd_rn(x, log1pf(expf(-x))) : log1pf(expf(x));
}

// Decay alpha = exp(g), g = -A * softplus(a + dt_bias), with A = exp(A_log)
// evaluated once per head by the caller.
__device__ __forceinline__ float gate_decay_scaled(float a, float A, float dt_bias) {
  float g = -__fmul_rn(A, softplus(__fadd_rn(a, dt_bias)));
  return expf(g);
}
// Decay alpha = exp(g), g = -exp(A_log) * softplus(a + dt_bias).
__device__ __forceinline__ float gate_decay(float a, float A_log, float dt_bias) {
  return gate_decay_scaled(a, expf(A_log), dt_bias);
}

// Write strength beta = sigmoid(b).
__device__ __forceinline__ float gate_beta(float b) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-b)));
}

// ------------------------------------------------------ element loads
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Four consecutive elements starting at p (16-byte aligned for fp32,
// 8-byte aligned for bf16), widened exactly to fp32.
__device__ __forceinline__ void load4(const float* p, float (&x)[4]) {
  float4 t = *reinterpret_cast<const float4*>(p);
  x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&x)[4]) {
  uint2 t = *reinterpret_cast<const uint2*>(p);
  x[0] = bf16_bits_to_float(t.x & 0xffffu);
  x[1] = bf16_bits_to_float(t.x >> 16);
  x[2] = bf16_bits_to_float(t.y & 0xffffu);
  x[3] = bf16_bits_to_float(t.y >> 16);
}
// A 16-byte piece of elements widened exactly to fp32: four fp32 values, or
// eight bf16 values (lower half-word first).
__device__ __forceinline__ void widen16(const uint4& t, float (&x)[4]) {
  x[0] = __uint_as_float(t.x); x[1] = __uint_as_float(t.y);
  x[2] = __uint_as_float(t.z); x[3] = __uint_as_float(t.w);
}
__device__ __forceinline__ void widen16(const uint4& t, float (&x)[8]) {
  const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16_bits_to_float(w[i] & 0xffffu);
    x[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
}
__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) {
  return bf16_bits_to_float(*reinterpret_cast<const unsigned short*>(p));
}

// State loads bypass L1 (ld.global.cg): a state tile is read once.
__device__ __forceinline__ void load_state4(const float* p, float (&x)[4]) {
  float4 t = __ldcg(reinterpret_cast<const float4*>(p));
  x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
}
__device__ __forceinline__ void load_state4(const __nv_bfloat16* p, float (&x)[4]) {
  uint2 t = __ldcg(reinterpret_cast<const uint2*>(p));
  x[0] = bf16_bits_to_float(t.x & 0xffffu);
  x[1] = bf16_bits_to_float(t.x >> 16);
  x[2] = bf16_bits_to_float(t.y & 0xffffu);
  x[3] = bf16_bits_to_float(t.y >> 16);
}

// Round-to-nearest-even to bf16, the single rounding of a stored state.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return a | (b << 16);
}

__device__ __forceinline__ void store_state4(float* p, const float (&x)[4]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
}
__device__ __forceinline__ void store_state4(__nv_bfloat16* p, const float (&x)[4]) {
  uint2 t;
  t.x = pack_bf16x2(x[0], x[1]);
  t.y = pack_bf16x2(x[2], x[3]);
  __stcs(reinterpret_cast<uint2*>(p), t);
}

// ------------------------------------------------ packed fp32 pairs (sm_100+)
// Two floats in one 64-bit register, operated on by the packed fp32
// instructions (mul.rn.f32x2 / fma.rn.f32x2 / add.rn.f32x2).  Each lane is
// rounded exactly as the scalar __fmul_rn / __fmaf_rn / __fadd_rn would
// round it, so packing changes the instruction count, never a result.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(f32x2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Four consecutive fp32 state elements as two pairs, bypassing L1.
__device__ __forceinline__ void load_state_pairs(const float* p, f32x2& a, f32x2& b) {
  asm("ld.global.cg.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}
__device__ __forceinline__ void load_state_pairs(const __nv_bfloat16* p, f32x2& a, f32x2& b) {
  float x[4];
  load_state4(p, x);
  a = pack2(x[0], x[1]);
  b = pack2(x[2], x[3]);
}
// Store two pairs as four consecutive state elements (bf16: rounded once).
__device__ __forceinline__ void store_state_pairs(float* p, f32x2 a, f32x2 b) {
  asm volatile("st.global.cs.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void store_state_pairs(__nv_bfloat16* p, f32x2 a, f32x2 b) {
  const float2 x = unpack2(a), y = unpack2(b);
  const float v[4] = {x.x, x.y, y.x, y.y};
  store_state4(p, v);
}
// The commit's fold on a pair: fma(u, khat, S * alpha) per lane.
__device__ __forceinline__ f32x2 fold2(f32x2 s, f32x2 alpha, f32x2 u, f32x2 kh) {
  return fma2(u, kh, mul2(s, alpha));
}

// --------------------------------------------------------- the recurrence
// One element's decay-then-write, the commit's fold and the verify's state
// update: S = fma(u, khat, S * alpha).
__device__ __forceinline__ float fold(float s, float alpha, float u, float kh) {
  return __fmaf_rn(u, kh, __fmul_rn(s, alpha));
}

// ----------------------------------------------------------- row planning
// Row plan shared by the kernels: checks a row against the documented
// contract, in the same order the error bits are documented.
struct SourceSlot {
  int slot;  // >= 0 live, -1 null row
  int err;   // GDN_ROW_ERR_* bits, 0 if fine
};

constexpr int kOutsideTable = INT_MIN;

// Slot holding the state after x folded tokens (block_size == 0: column 0).
// Returns kOutsideTable when the column lies outside the table.
__device__ __forceinline__ int slot_after(const int32_t* row, int stride,
                                          int block_size, long long x) {
  if (block_size == 0) return row[0];
  if (x < 1) return kOutsideTable;
  long long col = (x - 1) / block_size;
  if (col >= stride) return kOutsideTable;
  return row[col];
}

// The row's scalars a plan needs, requested together at the start of a
// kernel (each is in bounds for any row r < batch), so the plan costs one
// memory round trip instead of a chain of dependent ones.
struct RowScalars {
  int w;          // window_len[r]
  int slot0;      // slot_table[r][0]
  long long sp;   // seq_pos[r] (align mode), else 0
};
__device__ __forceinline__ RowScalars row_scalars(const int32_t* window_len, const int32_t* trow,
                                                  const int32_t* seq_pos, int block_size, int r) {
  RowScalars x;
  x.w = window_len[r];
  x.slot0 = trow[0];
  x.sp = block_size > 0 ? seq_pos[r] : 0;
  return x;
}

__device__ __forceinline__ SourceSlot source_slot(const RowScalars& x, int W, const int32_t* row,
                                                  int stride, int block_size, int num_slots) {
  SourceSlot s{-1, 0};
  const int w = x.w;
  if (w < 0 || w > W) { s.err = GDN_ROW_ERR_WINDOW; return s; }
  if (w == 0) return s;
  const long long p0 = x.sp;
  if (block_size > 0 && p0 < 1) { s.err = GDN_ROW_ERR_SEQPOS; return s; }
  int slot = block_size == 0 ? x.slot0 : slot_after(row, stride, block_size, p0);
  if (slot == kOutsideTable) { s.err = GDN_ROW_ERR_BLOCK; return s; }
  if (slot < -1 || slot >= num_slots) { s.err = GDN_ROW_ERR_SLOT; return s; }
  s.slot = slot;
  return s;
}

// Commit plan of one request row: checkpoint slot, final slot, accepted
// length and row errors, in the documented order of checks.  trow is the
// row of the layer's slot table, NULL for a layer with a bad group id.
// Boundary slots are validated here and looked up again when written.
struct RowCommit {
  int err;       // GDN_ROW_ERR_* bits
  bool live;     // something to fold and store
  int src, fin;  // checkpoint slot, final slot
  int n;         // accepted tokens
  long long p0;  // tokens already in the checkpoint (align mode)
};

__device__ __forceinline__ RowScalars row_scalars_from(int w, const int32_t* trow,
                                                       const int32_t* seq_pos, int block_size,
                                                       int r) {
  RowScalars x;
  x.w = w;
  x.slot0 = trow[0];
  x.sp = block_size > 0 ? seq_pos[r] : 0;
  return x;
}

__device__ __forceinline__ RowCommit row_commit_plan(int w, int n, const int32_t* trow,
                                                     int stride, int block_size,
                                                     const int32_t* seq_pos, int r,
                                                     int num_slots, int W) {
  RowCommit c{0, false, -1, -1, 0, 0};
  if (trow == nullptr) { c.err = GDN_ROW_ERR_GROUP; return c; }
  const RowScalars x = row_scalars_from(w, trow, seq_pos, block_size, r);
  SourceSlot src = source_slot(x, W, trow, stride, block_size, num_slots);
  if (src.err) { c.err = src.err; return c; }
  if (n < 0 || n > w) { c.err = GDN_ROW_ERR_ACCEPTED; return c; }
  if (src.slot < 0 || n == 0) return c;
  const long long p0 = block_size > 0 ? seq_pos[r] : 0;
  const int fin = slot_after(trow, stride, block_size, p0 + n);
  if (fin == kOutsideTable || fin == -1) { c.err = GDN_ROW_ERR_BLOCK; return c; }
  if (fin < -1 || fin >= num_slots) { c.err = GDN_ROW_ERR_SLOT; return c; }
  if (block_size > 0) {
    for (int j = 1; j < n; ++j) {
      if ((p0 + j) % block_size != 0) continue;
      const int bs = slot_after(trow, stride, block_size, p0 + j);
      if (bs == kOutsideTable || bs == -1) { c.err = GDN_ROW_ERR_BLOCK; return c; }
      if (bs < -1 || bs >= num_slots) { c.err = GDN_ROW_ERR_SLOT; return c; }
    }
  }
  c.live = true;
  c.src = src.slot;
  c.fin = fin;
  c.n = n;
  c.p0 = p0;
  return c;
}

}  // namespace gdn
