// gdn_conv.cu -- short-conv state commit over all layers in one launch.
//
// A GDN layer's causal depthwise convolution of width SL + 1 keeps, per
// slot and channel, the last SL convolution inputs (oldest first).  After
// sampling, that state must advance by the accepted tokens exactly as the
// recurrent state does, with the same plan (vLLM PR "[Spec Decode][Qwen4Exp]
// RecoverSSM for Qwen GDN and the PLE short conv", Purpose: the short conv
// "compacts its accepted window with the same plan"; Commits item 1: plan,
// conv and state steps of the commit).  The state after x folded tokens is
// the last SL entries of (checkpoint state ++ the row's first x inputs),
// written to the final slot and, in align mode, to every boundary slot.
//
// Pure data movement: every stored element is a copy of an input element,
// so results are bit-exact by construction.  One thread per channel: it
// loads its channel's whole checkpoint state into registers before writing
// anything, so a boundary slot equal to the checkpoint slot cannot be read
// after it has been overwritten.
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {

constexpr int kConvThreads = 256;
constexpr int kMaxConvState = 8;

template <typename T>
__global__ void __launch_bounds__(kConvThreads) gdn_conv_commit_kernel(const ConvParams p) {
  const int r = blockIdx.y, layer = blockIdx.z;
  const int c = blockIdx.x * kConvThreads + threadIdx.x;

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
  if (!plan.live || c >= p.C) return;

  const int SL = p.SL;
  T* pool = static_cast<T*>(p.pools[layer]);
  const T* in = static_cast<const T*>(p.inputs[layer]);
  const T* src = pool + ((size_t)plan.src * p.C + c) * SL;
  T old[kMaxConvState];
#pragma unroll
  for (int j = 0; j < kMaxConvState; ++j)
    if (j < SL) old[j] = src[j];

  // sequence element i: i < SL from the checkpoint, else input row i - SL
  auto element = [&](int i) -> T {
    T v = old[0];
#pragma unroll
    for (int j = 1; j < kMaxConvState; ++j)
      if (i == j) v = old[j];
    return i < SL ? v : in[(t0 + i - SL) * p.in_stride + c];
  };
  auto store_after = [&](int x, int slot) {
    T* dst = pool + ((size_t)slot * p.C + c) * SL;
    for (int j = 0; j < SL; ++j) dst[j] = element(x + j);
  };
  if (p.block_size > 0) {
    for (int x = 1; x < plan.n; ++x) {
      const long long pos = plan.p0 + x;
      if (pos % p.block_size == 0)
        store_after(x, slot_after(trow, p.table_stride, p.block_size, pos));
    }
  }
  store_after(plan.n, plan.fin);
}

int launch_conv_commit(const ConvParams& p, int dtype, cudaStream_t stream) {
  dim3 grid((p.C + kConvThreads - 1) / kConvThreads, p.batch, p.num_layers);
  if (dtype == GDN_DTYPE_BF16)
    gdn_conv_commit_kernel<unsigned short><<<grid, kConvThreads, 0, stream>>>(p);
  else
    gdn_conv_commit_kernel<unsigned int><<<grid, kConvThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
