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
// rank-1 updates from a ~1 KB-per-token record, write 64 KiB.  A thread
// holds 16-byte chunks c, c + NT, c + 2 NT, ... of a state tile in
// registers (NT threads), so every warp access is a run of whole 128-byte
// lines and each chunk's column block is fixed per thread.
//
// Ordering: each thread reads each of its chunks exactly once, before it
// writes anything, and writes only those same positions (in the boundary
// and final slots).  A boundary slot that equals the checkpoint slot is
// therefore never read after it has been overwritten, which is the
// guarantee "final folds before boundary folds" gives in a split commit.
//
// fp32 states: one CTA per (layer, row, head, 64-row tile): the record of
// the accepted tokens is staged with per-thread asynchronous copies
// (cp.async) issued ahead of the tile's loads, so four CTAs per SM keep
// ~128 KiB in flight.  bf16 states (gdn_commit_staged_kernel): one CTA per
// whole head, the tile itself copied into shared memory with the record and
// folded four chunks at a time, so four CTAs per SM again keep 128 KiB in
// flight (a register-held bf16 tile would keep only half of that).  The
// tile arrives in two commit groups, one per fold group, and the first is
// folded while the second is still landing.
//
// Ordering: in both kernels every chunk of the tile is read before any of
// it is written.
//
// Per-channel (KDA) records carry K gates per token; the fold then scales
// each column by its own gate, S[i][j] = fma(u[i], khat[j], S[i][j] *
// alpha[j]), in the same kernels (a compile-time flag).
//
// Rows the verify rejected (token rows out of range, or any other row
// error) carry the reject marker in gate record position 0; both kernels
// check it once the record is staged and store nothing for such a row, so
// a caller that replays verify and commit from one CUDA graph needs no host
// round trip to keep a stale record out of the state.
#include "gdn_async.cuh"
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {

// Waits until at most N of this thread's most recent cp.async commit groups
// are still in flight (a hardware wait, no polling).
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Slot-table row of request r for the group of `layer`, or NULL when the
// layer's group id is outside [0, num_groups).
__device__ __forceinline__ const int32_t* group_table_row(const CommitParams& p, int layer,
                                                          int r) {
  const int g = p.layer_group ? p.layer_group[layer] : 0;
  if (g < 0 || g >= p.num_groups) return nullptr;
  return p.slot_table + g * p.group_stride + (size_t)r * p.table_stride;
}

__device__ __forceinline__ RowCommit commit_row_plan(const CommitParams& p, int r,
                                                     const int32_t* trow) {
  return row_commit_plan(p.window_len[r], p.accepted_len[r], trow, p.table_stride,
                         p.block_size, p.seq_pos, r, p.num_slots, p.W);
}

// A 16-byte chunk of state (4 fp32 or 8 bf16) as packed fp32 pairs.
template <typename ST>
struct Chunk;
template <>
struct Chunk<float> {
  static constexpr int E = 4;
  static __device__ __forceinline__ void load(const float* p, f32x2 (&y)[2]) {
    load_state_pairs(p, y[0], y[1]);
  }
  static __device__ __forceinline__ void load_shared(const float* p, f32x2 (&y)[2]) {
    const ulonglong2 t = *reinterpret_cast<const ulonglong2*>(p);
    y[0] = t.x;
    y[1] = t.y;
  }
  static __device__ __forceinline__ void store(float* p, const f32x2 (&y)[2]) {
    store_state_pairs(p, y[0], y[1]);
  }
};
template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int E = 8;
  static __device__ __forceinline__ void widen(uint4 t, f32x2 (&y)[4]) {
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      y[i] = pack2(bf16_bits_to_float(w[i] & 0xffffu), bf16_bits_to_float(w[i] >> 16));
  }
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, f32x2 (&y)[4]) {
    widen(__ldcg(reinterpret_cast<const uint4*>(p)), y);
  }
  static __device__ __forceinline__ void load_shared(const __nv_bfloat16* p, f32x2 (&y)[4]) {
    widen(*reinterpret_cast<const uint4*>(p), y);
  }
  // Two fp32 values rounded to nearest even into one bf16 pair by a single
  // packed conversion (the same rounding as two scalar conversions).
  static __device__ __forceinline__ uint32_t round_pair(f32x2 v) {
    const float2 f = unpack2(v);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y), "f"(f.x));  // high <- y, low <- x
    return r;
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const f32x2 (&y)[4]) {
    const uint4 t = make_uint4(round_pair(y[0]), round_pair(y[1]), round_pair(y[2]), round_pair(y[3]));
    __stcs(reinterpret_cast<uint4*>(p), t);
  }
};

// Fold token t of a staged record into the thread's chunks.  u_s holds the
// corrections of rows [row_base, row_base + u_stride) of each token; g_s
// the gates, one per token ([W]) or, with the per-channel decay (KDA), one
// vector per token ([W][K]) whose entries scale the matching columns.
template <int K, typename ST, int M, int NT, bool KDA>
__device__ __forceinline__ void fold_token(f32x2 (&x)[M][Chunk<ST>::E / 2], const float* g_s,
                                           const float* k_s, const float* u_s, int t,
                                           int u_stride, int col, int c0, int row_base,
                                           int nchunks) {
  constexpr int E = Chunk<ST>::E;
  constexpr int CPR = K / E;
  f32x2 al2[E / 2];
  f32x2 kk[E / 2];
#pragma unroll
  for (int e = 0; e < E / 2; ++e) {
    kk[e] = *reinterpret_cast<const f32x2*>(k_s + t * K + col + 2 * e);
    al2[e] = KDA ? *reinterpret_cast<const f32x2*>(g_s + t * K + col + 2 * e)
                 : pack2(g_s[t], g_s[t]);
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int c = c0 + NT * m;
    if (c < nchunks) {
      const float u = u_s[t * u_stride + c / CPR - row_base];
      const f32x2 u2 = pack2(u, u);
#pragma unroll
      for (int e = 0; e < E / 2; ++e) x[m][e] = fold2(x[m][e], al2[e], u2, kk[e]);
    }
  }
}

template <typename ST, int M, int NT>
__device__ __forceinline__ void store_chunks(ST* dst, const f32x2 (&x)[M][Chunk<ST>::E / 2],
                                             int c0, int nchunks) {
  constexpr int E = Chunk<ST>::E;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int c = c0 + NT * m;
    if (c < nchunks) Chunk<ST>::store(dst + (size_t)c * E, x[m]);
  }
}

// ---------------------------------------------------------------------------
// One CTA per (layer, row, head, row tile).  Tile = NT * M chunks.  The
// record of the accepted tokens (u for the tile's rows, khat, alpha) is
// requested first and the tile's chunks right after, so the staging barrier
// waits only for the small record while the tile is still in flight.
constexpr int kCommitThreads = 256;

template <int K, typename ST, int M, bool KDA>
__global__ void __launch_bounds__(kCommitThreads)
    gdn_commit_kernel(const CommitParams p, int tiles_log2) {
  using C = Chunk<ST>;
  constexpr int E = C::E;
  constexpr int CPR = K / E;
  constexpr int NT = kCommitThreads;
  constexpr int TILE_ROWS = NT * M / CPR;
  extern __shared__ float smem[];

  const int tile = blockIdx.x & ((1 << tiles_log2) - 1);
  const int h = blockIdx.x >> tiles_log2;
  const int r = blockIdx.y, layer = blockIdx.z;
  const int tid = threadIdx.x;

  const int32_t* trow = group_table_row(p, layer, r);
  const RowCommit plan = commit_row_plan(p, r, trow);
  if (plan.err) {
    if (p.err && tid == 0 && tile == 0 && h == 0) atomicOr(p.err, plan.err);
    return;
  }
  if (!plan.live) return;  // null row or nothing accepted
  const int n = plan.n;
  const int row_base = tile * TILE_ROWS;
  const int rows = min(TILE_ROWS, p.V - row_base);
  if (rows <= 0) return;

  // ---- record first, as asynchronous copies: u [n][rows], khat [n][K],
  // ---- alpha [n] (rows and K are multiples of 16: whole 16-byte pieces)
  float* u_s = smem;                     // [W][TILE_ROWS]
  float* k_s = u_s + p.W * TILE_ROWS;    // [W][K]
  float* g_s = k_s + p.W * K;            // [W], or [W][K] for the per-channel gate
  const size_t rec = ((size_t)r * p.HV + h) * p.W;
  const float* ru = p.rec_u[layer] + rec * p.V + row_base;
  const float* rk = p.rec_k[layer] + rec * K;
  const float* rg = p.rec_g[layer] + rec * (KDA ? K : 1);
  const int urow4 = rows / 4;
  for (int i = tid; i < n * urow4; i += NT)
    cp_async16(u_s + (i / urow4) * TILE_ROWS + 4 * (i % urow4), ru + (size_t)(i / urow4) * p.V + 4 * (i % urow4));
  for (int i = tid; i < n * (K / 4); i += NT) cp_async16(k_s + 4 * i, rk + 4 * i);
  if constexpr (KDA) {
    for (int i = tid; i < n * (K / 4); i += NT) cp_async16(g_s + 4 * i, rg + 4 * i);
  } else {
    if (tid < n) cp_async4(g_s + tid, rg + tid);
  }
  cp_async_commit();

  // ---- then every chunk of the tile
  const size_t head = (size_t)p.V * K;
  ST* pool = static_cast<ST*>(p.pools[layer]);
  const ST* S0 = pool + ((size_t)plan.src * p.HV + h) * head;
  const int nchunks = (row_base + rows) * CPR;  // end of this tile's chunks in the head
  const int c0 = row_base * CPR + tid;
  f32x2 x[M][E / 2];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const int c = c0 + NT * m;
    if (c < nchunks) C::load(S0 + (size_t)c * E, x[m]);
  }
  cp_async_wait_all();
  __syncthreads();
  if (g_s[0] < 0.f) {  // the verify rejected this row: nothing is stored
    if (p.err && tid == 0 && tile == 0 && h == 0) atomicOr(p.err, GDN_ROW_ERR_REJECTED);
    return;
  }

  const int col = (tid % CPR) * E;  // fixed column block of this thread
  for (int t = 0; t < n; ++t) {
    fold_token<K, ST, M, NT, KDA>(x, g_s, k_s, u_s, t, TILE_ROWS, col, c0, row_base, nchunks);
    // align mode: the state after token p lands in slot(p) when p closes a block
    const long long pos = plan.p0 + t + 1;
    if (p.block_size > 0 && t + 1 < n && pos % p.block_size == 0) {
      const int bs = slot_after(trow, p.table_stride, p.block_size, pos);
      store_chunks<ST, M, NT>(pool + ((size_t)bs * p.HV + h) * head, x, c0, nchunks);
    }
  }
  store_chunks<ST, M, NT>(pool + ((size_t)plan.fin * p.HV + h) * head, x, c0, nchunks);
}

// bf16 states: a tile's widened fp32 values take twice the registers of its
// bytes, which caps the bytes a register-held tile keeps in flight.  Here the
// whole tile (a 128-row head) is first copied into shared memory by
// asynchronous copies, together with the record, and then folded G chunks
// at a time in registers; each element sees the same operations in the same
// order as in gdn_commit_kernel, and every chunk is read before any chunk of
// the tile is written, so a boundary or final slot equal to the source is
// still safe.
template <int K, typename ST, int M, int G, bool KDA, bool FULL>
__global__ void __launch_bounds__(kCommitThreads, 4)
    gdn_commit_staged_kernel(const CommitParams p, int tiles_log2) {
  using C = Chunk<ST>;
  constexpr int E = C::E;
  constexpr int CPR = K / E;
  constexpr int NT = kCommitThreads;
  constexpr int TILE_ROWS = NT * M / CPR;
  extern __shared__ __align__(16) float smem[];

  const int tile = blockIdx.x & ((1 << tiles_log2) - 1);
  const int h = blockIdx.x >> tiles_log2;
  const int r = blockIdx.y, layer = blockIdx.z;
  const int tid = threadIdx.x;

  const int32_t* trow = group_table_row(p, layer, r);
  const RowCommit plan = commit_row_plan(p, r, trow);
  if (plan.err) {
    if (p.err && tid == 0 && tile == 0 && h == 0) atomicOr(p.err, plan.err);
    return;
  }
  if (!plan.live) return;
  const int n = plan.n;
  const int row_base = tile * TILE_ROWS;
  const int rows = min(TILE_ROWS, p.V - row_base);
  if (rows <= 0) return;

  float* u_s = smem;                     // [W][TILE_ROWS]
  float* k_s = u_s + p.W * TILE_ROWS;    // [W][K]
  float* g_s = k_s + p.W * K;            // [W], or [W][K] for the per-channel gate
  ST* tile_s = reinterpret_cast<ST*>(g_s + ((p.W * (KDA ? K : 1) + 3) & ~3));  // [rows][K], 16-byte aligned
  const size_t rec = ((size_t)r * p.HV + h) * p.W;
  const float* ru = p.rec_u[layer] + rec * p.V + row_base;
  const float* rk = p.rec_k[layer] + rec * K;
  const float* rg = p.rec_g[layer] + rec * (KDA ? K : 1);
  const int urow4 = rows / 4;
  for (int i = tid; i < n * urow4; i += NT)
    cp_async16(u_s + (i / urow4) * TILE_ROWS + 4 * (i % urow4), ru + (size_t)(i / urow4) * p.V + 4 * (i % urow4));
  for (int i = tid; i < n * (K / 4); i += NT) cp_async16(k_s + 4 * i, rk + 4 * i);
  if constexpr (KDA) {
    for (int i = tid; i < n * (K / 4); i += NT) cp_async16(g_s + 4 * i, rg + 4 * i);
  } else {
    if (tid < n) cp_async4(g_s + tid, rg + tid);
  }
  const size_t head = (size_t)p.V * K;
  ST* pool = static_cast<ST*>(p.pools[layer]);
  const ST* S0 = pool + ((size_t)plan.src * p.HV + h) * head + (size_t)row_base * K;
  // the tile in M / G commit groups, one per fold group: a thread copies
  // exactly the chunks it later folds, so each group needs only the
  // thread's own wait, and a group is folded while the later ones land
  static_assert(M / G <= 2, "at most two fold groups per thread");
#pragma unroll
  for (int grp = 0; grp < M / G; ++grp) {
#pragma unroll
    for (int m = 0; m < G; ++m) {
      const int c = tid + NT * (G * grp + m);  // chunk inside the tile
      if (FULL || c < rows * CPR) cp_async16(tile_s + (size_t)c * E, S0 + (size_t)c * E);
    }
    cp_async_commit();
  }
  cp_async_wait_group<M / G - 1>();  // the record and the first fold group
  __syncthreads();
  if (g_s[0] < 0.f) {  // the verify rejected this row: nothing is stored
    if (p.err && tid == 0 && tile == 0 && h == 0) atomicOr(p.err, GDN_ROW_ERR_REJECTED);
    cp_async_wait_all();
    return;
  }

  // FULL: the head is a whole number of tiles, so every chunk a thread
  // names exists and no per-chunk guard is needed
  const int nchunks = (row_base + rows) * CPR;  // end of this tile's chunks in the head
  const int col = (tid % CPR) * E;
  const size_t fin_off = ((size_t)plan.fin * p.HV + h) * head;
#pragma unroll 1
  for (int grp = 0; grp < M / G; ++grp) {
    if (grp > 0) cp_async_wait_all();  // the second fold group's own chunks
    const int cg = row_base * CPR + tid + NT * G * grp;  // first chunk of this group (head index)
    f32x2 x[G][E / 2];
#pragma unroll
    for (int m = 0; m < G; ++m) {
      const int c = cg + NT * m;
      if (FULL || c < nchunks) C::load_shared(tile_s + (size_t)(c - row_base * CPR) * E, x[m]);
    }
    for (int t = 0; t < n; ++t) {
      f32x2 al2[E / 2], kk[E / 2];
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        kk[e] = *reinterpret_cast<const f32x2*>(k_s + t * K + col + 2 * e);
        al2[e] = KDA ? *reinterpret_cast<const f32x2*>(g_s + t * K + col + 2 * e)
                     : pack2(g_s[t], g_s[t]);
      }
#pragma unroll
      for (int m = 0; m < G; ++m) {
        if (FULL || cg + NT * m < nchunks) {
          const float u = u_s[t * TILE_ROWS + (cg + NT * m) / CPR - row_base];
          const f32x2 u2 = pack2(u, u);
#pragma unroll
          for (int e = 0; e < E / 2; ++e) x[m][e] = fold2(x[m][e], al2[e], u2, kk[e]);
        }
      }
      const long long pos = plan.p0 + t + 1;
      if (p.block_size > 0 && t + 1 < n && pos % p.block_size == 0) {
        const int bs = slot_after(trow, p.table_stride, p.block_size, pos);
        ST* dst = pool + ((size_t)bs * p.HV + h) * head;
#pragma unroll
        for (int m = 0; m < G; ++m) {
          const int c = cg + NT * m;
          if (FULL || c < nchunks) C::store(dst + (size_t)c * E, x[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < G; ++m) {
      const int c = cg + NT * m;
      if (FULL || c < nchunks) C::store(pool + fin_off + (size_t)c * E, x[m]);
    }
  }
}

// --------------------------------------------------------------- launchers
template <int K, typename ST, int M, bool KDA>
static int launch_commit_tiled_k(const CommitParams& p, cudaStream_t stream) {
  constexpr int CPR = K / Chunk<ST>::E;
  constexpr int TILE_ROWS = kCommitThreads * M / CPR;
  const int tiles = (p.V + TILE_ROWS - 1) / TILE_ROWS;
  int tiles_log2 = 0;
  while ((1 << tiles_log2) < tiles) ++tiles_log2;
  dim3 grid((unsigned)(p.HV << tiles_log2), p.batch, p.num_layers);
  const size_t smem = sizeof(float) * ((size_t)p.W * (TILE_ROWS + K) + (size_t)p.W * (KDA ? K : 1));
  auto kern = gdn_commit_kernel<K, ST, M, KDA>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  kern<<<grid, kCommitThreads, smem, stream>>>(p, tiles_log2);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// fp32 states: a tile is 64 state rows (8 chunks per thread for a 128-wide
// head): four such CTAs fit on an SM, and measured against whole-head and
// 32-row tiles, and against a persistent kernel streaming heads through
// shared memory with bulk asynchronous copies, it moves the most bytes.
template <int K, typename ST, bool KDA>
static int launch_commit_k(const CommitParams& p, cudaStream_t stream) {
  constexpr int CPR = K / Chunk<ST>::E;
  constexpr int MMAX = (128 * K) / Chunk<ST>::E / kCommitThreads;
  constexpr int MFULL = MMAX > 0 ? MMAX : 1;
  constexpr int M64 = (64 * CPR) / kCommitThreads;
  constexpr int M = M64 < 1 ? 1 : (M64 > MFULL ? MFULL : M64);
  return launch_commit_tiled_k<K, ST, M, KDA>(p, stream);
}

// bf16 states: whole 128-row heads staged in shared memory (see above).
template <int K, bool KDA>
static int launch_commit_bf16_k(const CommitParams& p, cudaStream_t stream) {
  using ST = __nv_bfloat16;
  constexpr int CPR = K / Chunk<ST>::E;
  constexpr int M = (128 * CPR) / kCommitThreads > 0 ? (128 * CPR) / kCommitThreads : 1;
  constexpr int G = M < 4 ? M : 4;
  constexpr int TILE_ROWS = kCommitThreads * M / CPR;
  const int tiles = (p.V + TILE_ROWS - 1) / TILE_ROWS;
  int tiles_log2 = 0;
  while ((1 << tiles_log2) < tiles) ++tiles_log2;
  dim3 grid((unsigned)(p.HV << tiles_log2), p.batch, p.num_layers);
  const size_t smem = sizeof(float) * ((size_t)p.W * (TILE_ROWS + K) +
                                       (((size_t)p.W * (KDA ? K : 1) + 3) & ~(size_t)3)) +
                      (size_t)TILE_ROWS * K * sizeof(ST);
  auto kern = p.V % TILE_ROWS == 0 ? gdn_commit_staged_kernel<K, ST, M, G, KDA, true>
                                    : gdn_commit_staged_kernel<K, ST, M, G, KDA, false>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  kern<<<grid, kCommitThreads, smem, stream>>>(p, tiles_log2);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <int K, bool KDA>
static int launch_commit_dtype(const CommitParams& p, bool bf, cudaStream_t stream) {
  return bf ? launch_commit_bf16_k<K, KDA>(p, stream) : launch_commit_k<K, float, KDA>(p, stream);
}

int launch_commit(const CommitParams& p, int head_k, int state_dtype, bool kda,
                  cudaStream_t stream) {
  const bool bf = state_dtype == GDN_DTYPE_BF16;
  switch (head_k) {
#define GDN_CASE(KK)                                                                  \
  case KK:                                                                            \
    return kda ? launch_commit_dtype<KK, true>(p, bf, stream)                         \
               : launch_commit_dtype<KK, false>(p, bf, stream);
    GDN_CASE(16)
    GDN_CASE(32)
    GDN_CASE(64)
    GDN_CASE(128)
#undef GDN_CASE
    default: return GDN_ERR_UNSUPPORTED;
  }
}

}  // namespace gdn
