// gdn_commit.cu -- all-layer replay commit in one launch.
//
// After sampling, each (layer, request row, value head) replays the first
// n = accepted_len tokens of its replay record onto the checkpoint,
//   S = fma(u_t, khat_t, S * alpha_t),  t = 0 .. n-1,
// and stores the state once into the row's final slot, plus the state at
// each block boundary crossed in align mode (tokenspeed PR "feat: add
// Qwen3.5 GDN ReplaySSM", Summary and Implementation; vLLM PR "[Spec
// Decode][Qwen4Exp] RecoverSSM for Qwen GDN and the PLE short conv",
// Purpose, Commits items 3 and 6, Test Result).
//
// The work is a pure stream: read a 64 KiB head (fp32, 128x128), fold a few
// rank-1 updates from a ~1 KB-per-token record, write 64 KiB.  One CTA of
// 256 threads owns a whole head; thread i holds the 16-byte chunks
// i, i + 256, i + 512, ... of it in registers, so every warp access is a
// run of whole 128-byte lines, and each chunk's column block is fixed per
// thread (256 is a multiple of the chunks per row).  The chunk loads are
// issued before the record is staged, so a CTA keeps its whole head in
// flight.
//
// Ordering: each thread reads each of its chunks exactly once, before it
// writes anything, and writes only those same positions (in the boundary
// and final slots).  A boundary slot that equals the checkpoint slot is
// therefore never read after it has been overwritten, which is the
// guarantee "final folds before boundary folds" gives in a split commit.
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {

constexpr int kCommitThreads = 256;

template <typename ST>
struct Chunk;
template <>
struct Chunk<float> {
  static constexpr int E = 4;  // elements per 16-byte chunk
  static __device__ __forceinline__ void load(const float* p, float (&x)[4]) {
    float4 t = __ldcg(reinterpret_cast<const float4*>(p));
    x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&x)[4]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
  }
};
template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int E = 8;
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[8]) {
    uint4 t = __ldcg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_bits_to_float(w[i] & 0xffffu);
      x[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&x)[8]) {
    uint4 t;
    t.x = pack_bf16x2(x[0], x[1]);
    t.y = pack_bf16x2(x[2], x[3]);
    t.z = pack_bf16x2(x[4], x[5]);
    t.w = pack_bf16x2(x[6], x[7]);
    __stcs(reinterpret_cast<uint4*>(p), t);
  }
};

template <int K, typename ST>
__global__ void __launch_bounds__(kCommitThreads, 2)
    gdn_commit_kernel(const CommitParams p) {
  using C = Chunk<ST>;
  constexpr int E = C::E;
  constexpr int CPR = K / E;                                   // chunks per state row
  constexpr int MAXM = (128 * K) / E / kCommitThreads;         // chunks per thread at V = 128
  constexpr int M = MAXM > 0 ? MAXM : 1;
  extern __shared__ float smem[];

  const int h = blockIdx.x, r = blockIdx.y, layer = blockIdx.z;
  const int tid = threadIdx.x;

  // ---- row plan (every thread evaluates it; the inputs are a few words)
  const int w = p.window_len[r];
  const int n = p.accepted_len[r];
  const int32_t* trow = p.slot_table + (size_t)r * p.table_stride;
  SourceSlot src = source_slot(w, p.W, trow, p.table_stride, p.block_size,
                               p.seq_pos, r, p.num_slots);
  int err = src.err;
  if (!err && (n < 0 || n > w)) err = GDN_ROW_ERR_ACCEPTED;
  const long long p0 = p.block_size > 0 && !err && src.slot >= 0 ? p.seq_pos[r] : 0;
  int fin = -1;
  if (!err && src.slot >= 0 && n > 0) {
    fin = slot_after(trow, p.table_stride, p.block_size, p0 + n);
    if (fin == kOutsideTable || fin == -1) err = GDN_ROW_ERR_BLOCK;
    else if (fin < -1 || fin >= p.num_slots) err = GDN_ROW_ERR_SLOT;
    if (!err && p.block_size > 0) {
      for (int j = 1; j < n; ++j) {
        if ((p0 + j) % p.block_size != 0) continue;
        const int bs = slot_after(trow, p.table_stride, p.block_size, p0 + j);
        if (bs == kOutsideTable || bs == -1) { err = GDN_ROW_ERR_BLOCK; break; }
        if (bs < -1 || bs >= p.num_slots) { err = GDN_ROW_ERR_SLOT; break; }
      }
    }
  }
  if (err) {
    if (p.err && tid == 0 && h == 0 && layer == 0) atomicOr(p.err, err);
    return;
  }
  if (src.slot < 0 || n == 0) return;  // null row or nothing accepted

  const size_t head = (size_t)p.V * K;
  ST* pool = static_cast<ST*>(p.pools[layer]);
  const ST* S0 = pool + ((size_t)src.slot * p.HV + h) * head;
  const int nchunks = p.V * CPR;

  // ---- issue every chunk load of the head
  float x[M][E];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int c = tid + kCommitThreads * m;
    if (c < nchunks) C::load(S0 + (size_t)c * E, x[m]);
  }

  // ---- stage the record of the accepted tokens: u [n][V], khat [n][K], alpha [n]
  float* u_s = smem;              // [W][V]
  float* k_s = u_s + p.W * p.V;   // [W][K]
  float* g_s = k_s + p.W * K;     // [W]
  const size_t rec = (((size_t)r * p.HV) + h) * p.W;
  const float* ru = p.rec_u[layer] + rec * p.V;
  const float* rk = p.rec_k[layer] + rec * K;
  const float* rg = p.rec_g[layer] + rec;
  for (int i = tid; i < n * p.V / 4; i += kCommitThreads)
    reinterpret_cast<float4*>(u_s)[i] = __ldg(reinterpret_cast<const float4*>(ru) + i);
  for (int i = tid; i < n * K / 4; i += kCommitThreads)
    reinterpret_cast<float4*>(k_s)[i] = __ldg(reinterpret_cast<const float4*>(rk) + i);
  if (tid < n) g_s[tid] = __ldg(rg + tid);
  __syncthreads();

  const int col = (tid % CPR) * E;  // fixed column block of this thread
  for (int t = 0; t < n; ++t) {
    const float al = g_s[t];
    float kk[E];
#pragma unroll
    for (int e = 0; e < E; ++e) kk[e] = k_s[t * K + col + e];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int c = tid + kCommitThreads * m;
      if (c < nchunks) {
        const float u = u_s[t * p.V + c / CPR];
#pragma unroll
        for (int e = 0; e < E; ++e) x[m][e] = fold(x[m][e], al, u, kk[e]);
      }
    }
    // align mode: the state after token p lands in slot(p) when p closes a block
    const long long pos = p0 + t + 1;
    if (p.block_size > 0 && t + 1 < n && pos % p.block_size == 0) {
      ST* dst = pool + ((size_t)slot_after(trow, p.table_stride, p.block_size, pos) * p.HV + h) * head;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int c = tid + kCommitThreads * m;
        if (c < nchunks) C::store(dst + (size_t)c * E, x[m]);
      }
    }
  }
  ST* dst = pool + ((size_t)fin * p.HV + h) * head;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int c = tid + kCommitThreads * m;
    if (c < nchunks) C::store(dst + (size_t)c * E, x[m]);
  }
}

template <int K, typename ST>
static int launch_commit_k(const CommitParams& p, cudaStream_t stream) {
  dim3 grid(p.HV, p.batch, p.num_layers);
  const size_t smem = sizeof(float) * (size_t)p.W * (p.V + K + 1);
  gdn_commit_kernel<K, ST><<<grid, kCommitThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int launch_commit(const CommitParams& p, int head_k, int state_dtype, cudaStream_t stream) {
  const bool bf = state_dtype == GDN_DTYPE_BF16;
  switch (head_k) {
    case 16: return bf ? launch_commit_k<16, __nv_bfloat16>(p, stream) : launch_commit_k<16, float>(p, stream);
    case 32: return bf ? launch_commit_k<32, __nv_bfloat16>(p, stream) : launch_commit_k<32, float>(p, stream);
    case 64: return bf ? launch_commit_k<64, __nv_bfloat16>(p, stream) : launch_commit_k<64, float>(p, stream);
    case 128: return bf ? launch_commit_k<128, __nv_bfloat16>(p, stream) : launch_commit_k<128, float>(p, stream);
    default: return GDN_ERR_UNSUPPORTED;
  }
}

size_t commit_smem_bytes(int head_k, int head_v, int W) {
  return sizeof(float) * (size_t)W * (head_v + head_k + 1);
}

}  // namespace gdn
