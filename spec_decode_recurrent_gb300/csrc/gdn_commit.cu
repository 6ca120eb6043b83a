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
#include <stdlib.h>

#include "gdn_async.cuh"
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {

constexpr int kCommitThreads = 256;

// Commit plan of one request row: checkpoint slot, final slot, accepted
// length and row errors, in the documented order of checks.  Boundary
// slots are validated here and looked up again when they are written.
struct RowCommit {
  int err;       // GDN_ROW_ERR_* bits
  bool live;     // something to fold and store
  int src, fin;  // checkpoint slot, final slot
  int n;         // accepted tokens
  long long p0;  // tokens already in the checkpoint (align mode)
};

__device__ __forceinline__ RowCommit commit_row_plan(const CommitParams& p, int r) {
  RowCommit c{0, false, -1, -1, 0, 0};
  const int w = p.window_len[r];
  const int n = p.accepted_len[r];
  const int32_t* trow = p.slot_table + (size_t)r * p.table_stride;
  SourceSlot src = source_slot(w, p.W, trow, p.table_stride, p.block_size, p.seq_pos, r,
                               p.num_slots);
  if (src.err) { c.err = src.err; return c; }
  if (n < 0 || n > w) { c.err = GDN_ROW_ERR_ACCEPTED; return c; }
  if (src.slot < 0 || n == 0) return c;
  const long long p0 = p.block_size > 0 ? p.seq_pos[r] : 0;
  const int fin = slot_after(trow, p.table_stride, p.block_size, p0 + n);
  if (fin == kOutsideTable || fin == -1) { c.err = GDN_ROW_ERR_BLOCK; return c; }
  if (fin < -1 || fin >= p.num_slots) { c.err = GDN_ROW_ERR_SLOT; return c; }
  if (p.block_size > 0) {
    for (int j = 1; j < n; ++j) {
      if ((p0 + j) % p.block_size != 0) continue;
      const int bs = slot_after(trow, p.table_stride, p.block_size, p0 + j);
      if (bs == kOutsideTable || bs == -1) { c.err = GDN_ROW_ERR_BLOCK; return c; }
      if (bs < -1 || bs >= p.num_slots) { c.err = GDN_ROW_ERR_SLOT; return c; }
    }
  }
  c.live = true;
  c.src = src.slot;
  c.fin = fin;
  c.n = n;
  c.p0 = p0;
  return c;
}

template <typename ST>
struct Chunk;
// A 16-byte chunk of state as packed fp32 pairs (E / 2 of them).
template <typename ST, int P>
__device__ __forceinline__ void pack_chunk(const float (&x)[2 * P], f32x2 (&y)[P]) {
#pragma unroll
  for (int i = 0; i < P; ++i) y[i] = pack2(x[2 * i], x[2 * i + 1]);
}
template <int P>
__device__ __forceinline__ void unpack_chunk(const f32x2 (&y)[P], float (&x)[2 * P]) {
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const float2 f = unpack2(y[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}
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
  static __device__ __forceinline__ void load_shared(const float* p, float (&x)[4]) {
    float4 t = *reinterpret_cast<const float4*>(p);
    x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
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
  static __device__ __forceinline__ void load_shared(const __nv_bfloat16* p, float (&x)[8]) {
    uint4 t = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = bf16_bits_to_float(w[i] & 0xffffu);
      x[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
    }
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
  const RowCommit plan = commit_row_plan(p, r);
  if (plan.err) {
    if (p.err && tid == 0 && h == 0 && layer == 0) atomicOr(p.err, plan.err);
    return;
  }
  if (!plan.live) return;  // null row or nothing accepted
  const int n = plan.n;
  const long long p0 = plan.p0;
  const int fin = plan.fin;
  const int32_t* trow = p.slot_table + (size_t)r * p.table_stride;

  const size_t head = (size_t)p.V * K;
  ST* pool = static_cast<ST*>(p.pools[layer]);
  const ST* S0 = pool + ((size_t)plan.src * p.HV + h) * head;
  const int nchunks = p.V * CPR;

  // ---- issue every chunk load of the head
  float x[M][E];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int c = tid + kCommitThreads * m;
    if (c < nchunks) C::load(S0 + (size_t)c * E, x[m]);
  }
  f32x2 xp[M][E / 2];

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

#pragma unroll
  for (int m = 0; m < M; ++m) pack_chunk<ST, E / 2>(x[m], xp[m]);
  const int col = (tid % CPR) * E;  // fixed column block of this thread
  for (int t = 0; t < n; ++t) {
    const f32x2 al2 = pack2(g_s[t], g_s[t]);
    f32x2 kk[E / 2];
#pragma unroll
    for (int e = 0; e < E / 2; ++e) kk[e] = *reinterpret_cast<const f32x2*>(k_s + t * K + col + 2 * e);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int c = tid + kCommitThreads * m;
      if (c < nchunks) {
        const float u = u_s[t * p.V + c / CPR];
        const f32x2 u2 = pack2(u, u);
#pragma unroll
        for (int e = 0; e < E / 2; ++e) xp[m][e] = fold2(xp[m][e], al2, u2, kk[e]);
      }
    }
    // align mode: the state after token p lands in slot(p) when p closes a block
    const long long pos = p0 + t + 1;
    if (p.block_size > 0 && t + 1 < n && pos % p.block_size == 0) {
      ST* dst = pool + ((size_t)slot_after(trow, p.table_stride, p.block_size, pos) * p.HV + h) * head;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int c = tid + kCommitThreads * m;
        float y[E];
        unpack_chunk<E / 2>(xp[m], y);
        if (c < nchunks) C::store(dst + (size_t)c * E, y);
      }
    }
  }
  ST* dst = pool + ((size_t)fin * p.HV + h) * head;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int c = tid + kCommitThreads * m;
    float y[E];
    unpack_chunk<E / 2>(xp[m], y);
    if (c < nchunks) C::store(dst + (size_t)c * E, y);
  }
}


// ---------------------------------------------------------------------------
// Pipelined form: a persistent CTA per SM streams heads through a ring of
// shared-memory stages.  Warp 0 (one elected lane) is the producer: for each
// live (layer, row, head) unit it waits for a free stage and issues bulk
// asynchronous copies (cp.async.bulk, TMA's untiled form) of the checkpoint
// head and of the accepted tokens' record into it, completing on the
// stage's "full" mbarrier.  Warps 1..8 are consumers: they wait for the
// stage, pull their 16-byte chunks into registers, fold the n tokens,
// release the stage and store from registers.  Two to four heads are in
// flight per SM at all times, independent of the folding work.
constexpr int kConsumerWarps = 8;
constexpr int kPipeThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxStages = 4;

template <int K, typename ST>
__global__ void __launch_bounds__(kPipeThreads, 1)
    gdn_commit_pipelined_kernel(const CommitParams p, int num_stages) {
  using C = Chunk<ST>;
  constexpr int E = C::E;
  constexpr int CPR = K / E;
  constexpr int NT = kConsumerWarps * 32;
  constexpr int MAXM = (128 * K) / E / NT;
  constexpr int M = MAXM > 0 ? MAXM : 1;
  extern __shared__ __align__(128) unsigned char smem_raw[];

  const int V = p.V;
  const uint32_t state_bytes = (uint32_t)(V * K * sizeof(ST));
  const uint32_t u_bytes = (uint32_t)(p.W * V * 4), k_bytes = (uint32_t)(p.W * K * 4);
  const uint32_t stage_bytes = state_bytes + u_bytes + k_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + (size_t)num_stages * stage_bytes);
  uint64_t* empty = full + kMaxStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < num_stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  const long long units = (long long)p.num_layers * p.batch * p.HV;
  const int nchunks = V * CPR;
  const size_t head = (size_t)V * K;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    uint32_t it = 0;
    for (long long x = blockIdx.x; x < units; x += gridDim.x) {
      const int h = (int)(x % p.HV);
      const int r = (int)((x / p.HV) % p.batch);
      const int layer = (int)(x / ((long long)p.HV * p.batch));
      const RowCommit plan = commit_row_plan(p, r);
      if (plan.err) {
        if (p.err && h == 0 && layer == 0) atomicOr(p.err, plan.err);
        continue;
      }
      if (!plan.live) continue;
      const int s = (int)(it % (uint32_t)num_stages);
      const uint32_t round = it / (uint32_t)num_stages;
      if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1u)) {
        if (p.err) atomicOr(p.err, kErrTimeout);
        return;
      }
      unsigned char* st = smem_raw + (size_t)s * stage_bytes;
      const ST* S0 = static_cast<const ST*>(p.pools[layer]) + ((size_t)plan.src * p.HV + h) * head;
      const size_t rec = ((size_t)r * p.HV + h) * p.W;
      const uint32_t nu = (uint32_t)(plan.n * V * 4), nk = (uint32_t)(plan.n * K * 4);
      mbar_arrive_expect_tx(&full[s], state_bytes + nu + nk);
      bulk_g2s(st, S0, state_bytes, &full[s]);
      bulk_g2s(st + state_bytes, p.rec_u[layer] + rec * V, nu, &full[s]);
      bulk_g2s(st + state_bytes + u_bytes, p.rec_k[layer] + rec * K, nk, &full[s]);
      ++it;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ct = threadIdx.x - 32;
  const int col = (ct % CPR) * E;
  uint32_t it = 0;
  for (long long x = blockIdx.x; x < units; x += gridDim.x) {
    const int h = (int)(x % p.HV);
    const int r = (int)((x / p.HV) % p.batch);
    const int layer = (int)(x / ((long long)p.HV * p.batch));
    const RowCommit plan = commit_row_plan(p, r);
    if (plan.err || !plan.live) continue;
    const int s = (int)(it % (uint32_t)num_stages);
    const uint32_t round = it / (uint32_t)num_stages;
    if (!mbar_wait(&full[s], round & 1u)) {
      if (p.err && lane == 0) atomicOr(p.err, kErrTimeout);
      return;
    }
    const unsigned char* st = smem_raw + (size_t)s * stage_bytes;
    const ST* S = reinterpret_cast<const ST*>(st);
    const float* u_s = reinterpret_cast<const float*>(st + state_bytes);
    const float* k_s = reinterpret_cast<const float*>(st + state_bytes + u_bytes);
    const float* rg = p.rec_g[layer] + ((size_t)r * p.HV + h) * p.W;

    f32x2 xs[M][E / 2];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int c = ct + NT * m;
      float y[E];
      if (c < nchunks) C::load_shared(S + (size_t)c * E, y);
      pack_chunk<ST, E / 2>(y, xs[m]);
    }
    ST* pool = static_cast<ST*>(p.pools[layer]);
    const int32_t* trow = p.slot_table + (size_t)r * p.table_stride;
    for (int t = 0; t < plan.n; ++t) {
      const float al = __ldg(rg + t);
      const f32x2 al2 = pack2(al, al);
      f32x2 kk[E / 2];
#pragma unroll
      for (int e = 0; e < E / 2; ++e) kk[e] = *reinterpret_cast<const f32x2*>(k_s + t * K + col + 2 * e);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const int c = ct + NT * m;
        if (c < nchunks) {
          const float u = u_s[t * V + c / CPR];
          const f32x2 u2 = pack2(u, u);
#pragma unroll
          for (int e = 0; e < E / 2; ++e) xs[m][e] = fold2(xs[m][e], al2, u2, kk[e]);
        }
      }
      const long long pos = plan.p0 + t + 1;
      if (p.block_size > 0 && t + 1 < plan.n && pos % p.block_size == 0) {
        ST* dst = pool + ((size_t)slot_after(trow, p.table_stride, p.block_size, pos) * p.HV + h) * head;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const int c = ct + NT * m;
          float y[E];
          unpack_chunk<E / 2>(xs[m], y);
          if (c < nchunks) C::store(dst + (size_t)c * E, y);
        }
      }
    }
    // every shared-memory read of this stage is done: hand it back
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    ST* dst = pool + ((size_t)plan.fin * p.HV + h) * head;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const int c = ct + NT * m;
      float y[E];
      unpack_chunk<E / 2>(xs[m], y);
      if (c < nchunks) C::store(dst + (size_t)c * E, y);
    }
    ++it;
  }
}

template <int K, typename ST>
static int launch_commit_pipelined_k(const CommitParams& p, cudaStream_t stream) {
  static int num_sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 64 && num_sms[dev] == 0)
    cudaDeviceGetAttribute(&num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
  const int sms = dev < 64 && num_sms[dev] > 0 ? num_sms[dev] : 148;
  const size_t stage = (size_t)p.V * K * sizeof(ST) + (size_t)p.W * (p.V + K) * 4;
  const size_t bars = 2 * kMaxStages * sizeof(uint64_t);
  const size_t budget = 227 * 1024 - bars;
  int stages = (int)(budget / stage);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return GDN_ERR_UNSUPPORTED;
  const size_t smem = (size_t)stages * stage + bars;
  if (cudaFuncSetAttribute(gdn_commit_pipelined_kernel<K, ST>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  const long long units = (long long)p.num_layers * p.batch * p.HV;
  const int grid = (int)(units < sms ? units : sms);
  gdn_commit_pipelined_kernel<K, ST><<<grid, kPipeThreads, smem, stream>>>(p, stages);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
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
  static const char* variant = getenv("GDN_COMMIT_VARIANT");
  if (!(variant && variant[0] == 'r')) {
    switch (head_k) {
      case 16: return bf ? launch_commit_pipelined_k<16, __nv_bfloat16>(p, stream) : launch_commit_pipelined_k<16, float>(p, stream);
      case 32: return bf ? launch_commit_pipelined_k<32, __nv_bfloat16>(p, stream) : launch_commit_pipelined_k<32, float>(p, stream);
      case 64: return bf ? launch_commit_pipelined_k<64, __nv_bfloat16>(p, stream) : launch_commit_pipelined_k<64, float>(p, stream);
      case 128: return bf ? launch_commit_pipelined_k<128, __nv_bfloat16>(p, stream) : launch_commit_pipelined_k<128, float>(p, stream);
      default: return GDN_ERR_UNSUPPORTED;
    }
  }
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
