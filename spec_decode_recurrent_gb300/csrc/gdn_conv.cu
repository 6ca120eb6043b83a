// gdn_conv.cu -- short-conv state commit over all layers in one launch.
//
// A GDN layer's causal depthwise convolution of width SL + 1 keeps, per
// slot and channel, the last SL convolution inputs (oldest first).  After
// sampling, that state must advance by the accepted tokens exactly as the
// recurrent state does, with the same plan (vLLM PR "[Spec Decode][Qwen4Exp]
// RecoverSSM for Qwen GDN and the PLE short conv", Purpose: the conv state
// is advanced over the accepted tokens by the recurrent commit's plan;
// Commits item 1: plan, conv and state steps of the commit).  The state after x folded tokens is
// the last SL entries of (checkpoint state ++ the row's first x inputs),
// written to the final slot and, in align mode, to every boundary slot.
//
// Pure data movement: every stored element is a copy of an input element,
// so results are bit-exact by construction.  A thread loads its channels'
// whole checkpoint state into registers before writing anything and then
// shifts it token by token, so a boundary slot equal to the checkpoint slot
// cannot be read after it has been overwritten.
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {

constexpr int kConvThreads = 256;

// 32-bit word k of a 16-byte chunk (k a compile-time constant after unrolling).
__device__ __forceinline__ uint32_t chunk_word(const uint4& q, int k) {
  return k == 0 ? q.x : (k == 1 ? q.y : (k == 2 ? q.z : q.w));
}
// Element i of a chunk of 16-bit (B = 2) or 32-bit (B = 4) elements.
template <int B>
__device__ __forceinline__ uint32_t chunk_elem(const uint4& q, int i) {
  if (B == 4) return chunk_word(q, i);
  return (chunk_word(q, i >> 1) >> ((i & 1) * 16)) & 0xffffu;
}
template <int B, int NE>
__device__ __forceinline__ uint4 make_chunk(const uint32_t (&e)[NE], int k) {
  constexpr int E = 16 / B;
  if (B == 4) return make_uint4(e[k * E], e[k * E + 1], e[k * E + 2], e[k * E + 3]);
  return make_uint4(e[k * E] | (e[k * E + 1] << 16), e[k * E + 2] | (e[k * E + 3] << 16),
                    e[k * E + 4] | (e[k * E + 5] << 16), e[k * E + 6] | (e[k * E + 7] << 16));
}

// A thread owns one group of E = 16 / B channels (B = element bytes): their
// states are E * SL contiguous elements (SL 16-byte chunks) and each token
// row gives one 16-byte chunk of their inputs, so every access is a full
// 16 bytes.  Elements travel as raw bits in 32-bit registers.
template <int B, int SL>
__global__ void __launch_bounds__(kConvThreads) gdn_conv_commit_kernel(const ConvParams p) {
  constexpr int E = 16 / B;   // channels per thread
  constexpr int NE = E * SL;  // state elements per thread
  const int r = blockIdx.y, layer = blockIdx.z;
  const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * E;

  const int g = p.layer_group ? p.layer_group[layer] : 0;
  const int32_t* trow = (g < 0 || g >= p.num_groups)
                            ? nullptr
                            : p.slot_table + g * p.group_stride + (size_t)r * p.table_stride;
  RowCommit plan = row_commit_plan(p.window_len[r], p.accepted_len[r], trow, p.table_stride,
                                   p.block_size, p.seq_pos, r, p.num_slots, p.W);
  long long t0 = 0;
  if (!plan.err && plan.live) {
    t0 = p.token_start[r];
    if (t0 < 0 || t0 + p.window_len[r] > p.num_tokens) plan.err = GDN_ROW_ERR_TOKENS;
  }
  if (plan.err) {
    if (p.err && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, plan.err);
    return;
  }
  if (!plan.live || c0 >= p.C) return;

  unsigned char* pool = static_cast<unsigned char*>(p.pools[layer]);
  const unsigned char* in = static_cast<const unsigned char*>(p.inputs[layer]);
  // the checkpoint state of the group, element ch * SL + j, read before any
  // write; then one shift per accepted token: drop the oldest entry of each
  // channel and append the token's input
  uint32_t st[NE];
  {
    const uint4* src =
        reinterpret_cast<const uint4*>(pool + ((size_t)plan.src * p.C + c0) * SL * B);
#pragma unroll
    for (int k = 0; k < SL; ++k) {
      const uint4 q = __ldcg(src + k);
#pragma unroll
      for (int i = 0; i < E; ++i) st[k * E + i] = chunk_elem<B>(q, i);
    }
  }
  auto dst_of = [&](int slot) {
    return reinterpret_cast<uint4*>(pool + ((size_t)slot * p.C + c0) * SL * B);
  };
  for (int t = 0; t < plan.n; ++t) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(in + ((t0 + t) * p.in_stride + c0) * B));
#pragma unroll
    for (int ch = 0; ch < E; ++ch) {
#pragma unroll
      for (int j = 0; j + 1 < SL; ++j) st[ch * SL + j] = st[ch * SL + j + 1];
      st[ch * SL + SL - 1] = chunk_elem<B>(q, ch);
    }
    const long long pos = plan.p0 + t + 1;
    const bool boundary = p.block_size > 0 && t + 1 < plan.n && pos % p.block_size == 0;
    if (boundary || t + 1 == plan.n) {
      uint4* dst = dst_of(boundary ? slot_after(trow, p.table_stride, p.block_size, pos)
                                   : plan.fin);
#pragma unroll
      for (int k = 0; k < SL; ++k) __stcs(dst + k, make_chunk<B, NE>(st, k));
    }
  }
}

template <int B>
static int launch_conv_t(const ConvParams& p, cudaStream_t stream) {
  constexpr int E = 16 / B;
  const int groups = p.C / E;
  dim3 grid((groups + kConvThreads - 1) / kConvThreads, p.batch, p.num_layers);
  switch (p.SL) {
#define GDN_SL(N) \
  case N: gdn_conv_commit_kernel<B, N><<<grid, kConvThreads, 0, stream>>>(p); break;
    GDN_SL(1) GDN_SL(2) GDN_SL(3) GDN_SL(4) GDN_SL(5) GDN_SL(6) GDN_SL(7) GDN_SL(8)
#undef GDN_SL
    default: return GDN_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int launch_conv_commit(const ConvParams& p, int dtype, cudaStream_t stream) {
  if (dtype == GDN_DTYPE_BF16) return launch_conv_t<2>(p, stream);
  return launch_conv_t<4>(p, stream);
}

}  // namespace gdn
