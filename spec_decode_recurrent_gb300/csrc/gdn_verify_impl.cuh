// gdn_verify_impl.cuh -- speculative verify and native per-draft snapshot
// kernels (templates).  Each gdn_verify_k*.cu instantiates the head widths
// and gate kinds it names, so the instantiations compile in parallel;
// gdn_verify.cu dispatches a call to them.
//
// The window in matrix form.  With the checkpoint C and the gate products
// gamma_t = alpha_0 ... alpha_t and rho_{t,j} = alpha_{j+1} ... alpha_t
// (per channel for the KDA decay), the state after token t is
//   S_t = C diag(gamma_t) + sum_{j<=t} u_j (rho_{t,j} khat_j)^T,
// so the two products the recurrence needs from H_t = alpha_t S_{t-1} are
//   d_t = H_t khat_t = C kt_t + sum_{j<t}  A_{t,j} u_j,   kt_t = gamma_t khat_t,
//   o_t = S_t qhat_t = C qt_t + sum_{j<=t} B_{t,j} u_j,   qt_t = gamma_t qhat_t,
// with A_{t,j} = <rho_{t,j} khat_j, khat_t> and B_{t,j} = <rho_{t,j} khat_j,
// qhat_t>, and u_t = beta_t (v_t - d_t) (tokenspeed PR "feat: add Qwen3.5 GDN
// ReplaySSM", Summary; vLLM PR "[Spec Decode][Qwen4Exp] RecoverSSM for Qwen
// GDN and the PLE short conv", Purpose).  The same d_t, u_t and o_t as the
// token-by-token recurrence in exact arithmetic; what it changes is the
// work per state element: 2w products against the checkpoint, all
// independent, instead of a decay, two dot products and a rank-1 update per
// token in a serial chain.  The window's side (kt, qt, A, B: O(w^2 K)) is
// computed once per CTA.
//
// One CTA of 4 warps covers up to four tiles of VT state rows (64 for
// K = 128) of one (request row, value head), the tile held in registers, a
// cooperative 4-warp CTA per 128x128 state head (tokenspeed PR,
// Implementation).  Per tile and token each lane forms its partial products
// with kt_t and qt_t; the LPR lanes of a row combine them by recursive
// halving (each exchange sends half of the remaining values and keeps the
// other half), and the row sums land in shared memory.  After the last tile
// one thread per row runs the short scalar recurrence for u_t and o_t and
// writes both, coalesced.  Tiles reach the CTA as single bulk copies
// (cp.async.bulk, one thread per tile: 32 KiB for a 64 x 128 fp32 tile)
// into a shared buffer, completed
// through an mbarrier; tile i + 1 is requested as soon as every warp has
// moved tile i into registers.
//
// VERIFY mode writes o_t and the replay record (u_t, khat_t, alpha_t) and no
// state.  NATIVE mode (one tile per CTA) computes the same u_t and o_t the
// same way, then folds the tile token by token with the commit's update,
// S_t = fma(u_t, khat_t, S_{t-1} * alpha_t), and writes every S_t.  So the
// verify's outputs equal the native ones bit for bit, and a commit of n
// accepted tokens (the same fold over the verify's records) equals the
// native state after token n.
#pragma once

#include <type_traits>

#include "gdn_async.cuh"
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {

template <int K>
struct VerifyTile {
  static constexpr int LPR = K / 16;              // lanes per state row
  static constexpr int RPW = 32 / LPR;            // rows per warp per row group
  // four row groups per thread at K = 128: each token's key and query
  // values a lane reads from shared memory serve four rows (two measured
  // slower: the shared-memory data pipe was the busiest unit)
  static constexpr int RPT = (K == 128) ? 4 : 1;  // row groups per thread
  static constexpr int WARPS = 4;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int VT = WARPS * RPW * RPT;    // state rows per tile
  // CTAs per SM the registers must allow: four at K = 128 (four row groups
  // per thread, about 110 registers); otherwise six (80 registers) for the
  // verify with an fp32 state and seven (72) for the rest
  template <bool NATIVE, typename ST, bool KDA>
  static constexpr int min_ctas() {
    return K == 128 ? 4 : ((!NATIVE && sizeof(ST) == 4) ? 6 : 7);
  }
};

// Shared memory of one verify CTA covering NS tiles (SV = NS * VT staged
// value rows), as float offsets after the mbarrier (kBarBytes) and the tile
// buffer the bulk copies fill (NS > 1 only).  One buffer: two to four,
// each CTA streaming more tiles, measured slower on every workload (the
// shared memory they take costs resident CTAs).
constexpr int kBarBytes = 16;
template <int K, typename ST, bool KDA, bool NATIVE>
struct VerifySmem {
  int W, SV;
  __host__ __device__ constexpr VerifySmem(int W_, int NS)
      : W(W_), SV(NS * VerifyTile<K>::VT) {}
  __host__ __device__ constexpr size_t tile_bytes(int NS) const {
    return NS > 1 ? (size_t)VerifyTile<K>::VT * K * sizeof(ST) : 0;
  }
  __host__ __device__ constexpr int kt() const { return 0; }             // [W][K] gamma khat
  __host__ __device__ constexpr int qt() const { return W * K; }         // [W][K] gamma qhat
  __host__ __device__ constexpr int v() const { return 2 * W * K; }      // [W][SV] values
  __host__ __device__ constexpr int gs() const { return v() + W * SV; }  // [W][4] alpha, beta
  __host__ __device__ constexpr int ab() const { return gs() + 4 * W; }  // [2][W][W] A, B
  // A and B padded to whole 16-byte pieces: al is read and written in them
  __host__ __device__ constexpr int al() const { return ab() + ((2 * W * W + 3) & ~3); }  // [W][K] (KDA)
  // khat and qhat ([W][K] each) are read only while the window is staged
  // and, in the verify, share their space with the products C kt, C qt
  // ([W][2][SV]) and u ([W][SV]), which are written only after it; the
  // native kernel still folds with khat after its products, so there they
  // are separate
  __host__ __device__ constexpr int kh() const { return al() + (KDA ? W * K : 0); }
  __host__ __device__ constexpr int qh() const { return kh() + W * K; }
  __host__ __device__ constexpr int pq() const { return NATIVE ? qh() + W * K : kh(); }
  __host__ __device__ constexpr int u() const { return pq() + 2 * W * SV; }
  __host__ __device__ constexpr int floats() const {
    return (u() + W * SV) > (qh() + W * K) ? (u() + W * SV) : (qh() + W * K);
  }
  __host__ __device__ constexpr size_t bytes(int NS) const {
    return kBarBytes + tile_bytes(NS) + sizeof(float) * (size_t)floats();
  }
};

// A tile's checkpoint rows from the shared-memory tile buffer (a verbatim
// copy of VT contiguous state rows) into the register buffer.
template <int K>
__device__ __forceinline__ void load_tile_shared(f32x2 (&s)[VerifyTile<K>::RPT][8], const float* buf,
                                                 int warp, int l, int lr) {
  using Tile = VerifyTile<K>;
#pragma unroll
  for (int g = 0; g < Tile::RPT; ++g) {
    const int row = (g * Tile::WARPS + warp) * Tile::RPW + lr;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const ulonglong2 t = *reinterpret_cast<const ulonglong2*>(buf + row * K + 4 * (l + Tile::LPR * m));
      s[g][2 * m] = t.x;
      s[g][2 * m + 1] = t.y;
    }
  }
}
template <int K>
__device__ __forceinline__ void load_tile_shared(f32x2 (&s)[VerifyTile<K>::RPT][8],
                                                 const __nv_bfloat16* buf, int warp, int l, int lr) {
  using Tile = VerifyTile<K>;
#pragma unroll
  for (int g = 0; g < Tile::RPT; ++g) {
    const int row = (g * Tile::WARPS + warp) * Tile::RPW + lr;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint2 t = *reinterpret_cast<const uint2*>(buf + row * K + 4 * (l + Tile::LPR * m));
      s[g][2 * m] = pack2(bf16_bits_to_float(t.x & 0xffffu), bf16_bits_to_float(t.x >> 16));
      s[g][2 * m + 1] = pack2(bf16_bits_to_float(t.y & 0xffffu), bf16_bits_to_float(t.y >> 16));
    }
  }
}

// Checkpoint rows of one tile into a register buffer (zeros past V).
template <int K, typename ST, bool FULL>
__device__ __forceinline__ void load_tile(f32x2 (&s)[VerifyTile<K>::RPT][8], const ST* S0, int tile,
                                          int V, int warp, int l, int lr) {
  using Tile = VerifyTile<K>;
#pragma unroll
  for (int g = 0; g < Tile::RPT; ++g) {
    const int row = tile * Tile::VT + (g * Tile::WARPS + warp) * Tile::RPW + lr;
    if (FULL || row < V) {
#pragma unroll
      for (int m = 0; m < 4; ++m)
        load_state_pairs(S0 + (size_t)row * K + 4 * (l + Tile::LPR * m), s[g][2 * m], s[g][2 * m + 1]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) s[g][j] = 0ull;
    }
  }
}

// The index of the first value a lane holds after LaneHalve<OFF, N> (what
// LaneHalve accumulates in `base`, without the exchanges).
template <int OFF, int N>
struct LaneHalveIndex {
  static __device__ __forceinline__ int run(int l) {
    if constexpr (OFF >= 1 && N > 1)
      return ((l & OFF) != 0 ? N / 2 : 0) + LaneHalveIndex<OFF / 2, N / 2>::run(l);
    return 0;
  }
};

// One token's key and query L2-normalised by a whole warp: lane i < K / 4
// holds elements 4 i .. 4 i + 3 of each (zeros elsewhere) and writes its
// four normalised values into khat_row and qhat_row.
template <int K>
__device__ __forceinline__ void normalise_token(const float (&kx)[4], const float (&qx)[4],
                                                float* khat_row, float* qhat_row, int lane) {
  float ks = __fmul_rn(kx[0], kx[0]), qs = __fmul_rn(qx[0], qx[0]);
#pragma unroll
  for (int e = 1; e < 4; ++e) {
    ks = __fmaf_rn(kx[e], kx[e], ks);
    qs = __fmaf_rn(qx[e], qx[e], qs);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    ks = __fadd_rn(ks, __shfl_xor_sync(0xffffffffu, ks, off));
    qs = __fadd_rn(qs, __shfl_xor_sync(0xffffffffu, qs, off));
  }
  // x / sqrt(|x|^2 + eps) as x * rsqrt(|x|^2 + eps), rsqrt correctly rounded
  const float kr = __frsqrt_rn(__fadd_rn(ks, kL2NormEps));
  const float qr = __frsqrt_rn(__fadd_rn(qs, kL2NormEps));
  if (lane < K / 4) {
    *reinterpret_cast<float4*>(khat_row + 4 * lane) = make_float4(
        __fmul_rn(kx[0], kr), __fmul_rn(kx[1], kr), __fmul_rn(kx[2], kr), __fmul_rn(kx[3], kr));
    *reinterpret_cast<float4*>(qhat_row + 4 * lane) = make_float4(
        __fmul_rn(qx[0], qr), __fmul_rn(qx[1], qr), __fmul_rn(qx[2], qr), __fmul_rn(qx[3], qr));
  }
}

// Recursive halving of N per-lane values over the lanes of a row group: at
// lane distance OFF the lane with that bit set keeps the upper half of its
// values and sends the lower half, its partner the reverse, and each adds
// what it receives; with one value left the remaining distances are plain
// butterfly additions.  base accumulates the index of the lane's first
// remaining value.
template <int OFF, int N>
struct LaneHalve {
  template <int NV>
  static __device__ __forceinline__ void run(float (&x)[NV], int l, int& base) {
    if constexpr (OFF >= 1) {
      if constexpr (N > 1) {
        constexpr int H = N / 2;
        const bool up = (l & OFF) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const float send = up ? x[i] : x[i + H];
          const float keep = up ? x[i + H] : x[i];
          x[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, OFF));
        }
        if (up) base += H;
        LaneHalve<OFF / 2, H>::run(x, l, base);
      } else {
        x[0] = __fadd_rn(x[0], __shfl_xor_sync(0xffffffffu, x[0], OFF));
        LaneHalve<OFF / 2, 1>::run(x, l, base);
      }
    }
  }
};

// The window's side, from khat, qhat ([W][K]) and the gates (gs [W][4]
// alpha, beta; al [W][K] per channel with the KDA decay), by `nthreads`
// threads (`nwarps` whole warps):
//   channel c: gamma_t = gamma_{t-1} * alpha_t, kt_t = gamma_t khat_t,
//   qt_t = gamma_t qhat_t (one thread per channel);
//   A_{t,j} = <rho_{t,j} khat_j, khat_t> (j < t), B_{t,j} = <rho_{t,j}
//   khat_j, qhat_t> (j <= t): warp j (mod nwarps) walks t upward from j with
//   the running product rho per channel, each lane summing its channels
//   c = lane + 32 i in order; four tokens' eight sums at a time are then
//   summed over the warp's lanes by recursive halving (one chain of five
//   exchanges for all eight).
// The caller orders the inputs before and the outputs after (barriers).
template <int K, bool KDA>
__device__ __forceinline__ void window_side(int w, int W, const float* kh_s, const float* qh_s,
                                            const float* gs_s, const float* al_s, float* kt_s,
                                            float* qt_s, float* A_s, float* B_s, int tid,
                                            int nthreads, int warp, int nwarps, int lane) {
  auto decay_of = [&](int t, int c) { return KDA ? al_s[t * K + c] : gs_s[4 * t]; };
  for (int c = tid; c < K; c += nthreads) {
    float gam = 1.f;
    for (int t = 0; t < w; ++t) {
      gam = __fmul_rn(gam, decay_of(t, c));
      kt_s[t * K + c] = __fmul_rn(gam, kh_s[t * K + c]);
      qt_s[t * K + c] = __fmul_rn(gam, qh_s[t * K + c]);
    }
  }
  constexpr int CPL = (K + 31) / 32;  // channels per lane
  for (int j = warp; j < w; j += nwarps) {
    float kr[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      kr[i] = c < K ? kh_s[j * K + c] : 0.f;  // rho_{j,j} khat_j = khat_j
    }
    for (int tb = j; tb < w; tb += 4) {
      float x[8];
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const int t = tb + tt;
        float sa = 0.f, sb = 0.f;
        if (t < w) {
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = lane + 32 * i;
            if (c < K) {
              if (t > j) kr[i] = __fmul_rn(kr[i], decay_of(t, c));
              sa = __fmaf_rn(kr[i], kh_s[t * K + c], sa);
              sb = __fmaf_rn(kr[i], qh_s[t * K + c], sb);
            }
          }
        }
        x[2 * tt] = sa;
        x[2 * tt + 1] = sb;
      }
      int base = 0;
      LaneHalve<16, 8>::run(x, lane, base);  // one sum per lane, equal within groups of 4
      if ((lane & 3) == 0) {
        const int t = tb + (base >> 1);
        if (t < w) {
          if ((base & 1) == 0) {
            if (t > j) A_s[t * W + j] = x[0];
          } else {
            B_s[t * W + j] = x[0];
          }
        }
      }
    }
  }
}

// u_t and o_t of one row from its products pq ([W][2][SV], row `row`), its
// values vload(t) and the window's beta (gs) and A, B ([W][W]):
//   d = C kt + sum_{j<t} A u_j,  u = beta (v - d),  o = C qt + sum_{j<=t} B u_j.
// u_t lands in u_s[t][row]; o_t at optr[t * out_stride]; u_t also at
// uptr[t * V] when uptr is not null.  WC > 0: the record stride W is WC
// and the loops are unrolled, u_j kept in registers (the same operations in
// the same order).
template <int WC, typename VLoad>
__device__ __forceinline__ void row_recurrence(int row, int w, int W, int SV, const float* pq_s,
                                               float* u_s, const float* gs_s, const float* A_s,
                                               const float* B_s, VLoad vload, float* optr,
                                               long long out_stride, float* uptr, int V) {
  if constexpr (WC > 0) {
    float ur[WC];
#pragma unroll
    for (int t = 0; t < WC; ++t) {
      if (t < w) {
        float d = pq_s[(2 * t) * SV + row];
#pragma unroll
        for (int j = 0; j < t; ++j) d = __fmaf_rn(A_s[t * WC + j], ur[j], d);
        const float u = __fmul_rn(gs_s[4 * t + 1], __fsub_rn(vload(t), d));
        float o = pq_s[(2 * t + 1) * SV + row];
#pragma unroll
        for (int j = 0; j < t; ++j) o = __fmaf_rn(B_s[t * WC + j], ur[j], o);
        o = __fmaf_rn(B_s[t * WC + t], u, o);
        ur[t] = u;
        u_s[t * SV + row] = u;
        optr[t * out_stride] = o;
        if (uptr) uptr[(size_t)t * V] = u;
      }
    }
    return;
  }
  for (int t = 0; t < w; ++t) {
    float d = pq_s[(2 * t) * SV + row];
    for (int j = 0; j < t; ++j) d = __fmaf_rn(A_s[t * W + j], u_s[j * SV + row], d);
    const float u = __fmul_rn(gs_s[4 * t + 1], __fsub_rn(vload(t), d));
    float o = pq_s[(2 * t + 1) * SV + row];
    for (int j = 0; j < t; ++j) o = __fmaf_rn(B_s[t * W + j], u_s[j * SV + row], o);
    o = __fmaf_rn(B_s[t * W + t], u, o);
    u_s[t * SV + row] = u;
    optr[t * out_stride] = o;
    if (uptr) uptr[(size_t)t * V] = u;
  }
}

// Per token: the tile's rows against kt_t and qt_t, summed over each row's
// lanes, into pq_s[t][0 / 1][row0 + row].  Value v = 2 g + which of a lane
// is row group g's C kt (which 0) or C qt (which 1).  Which values a lane
// ends with, and where they go, is fixed per lane and worked out once.
// WC > 0: at most WC tokens, the token loop unrolled by two (fully unrolled
// it measured slower).
template <int K, int WC>
__device__ __forceinline__ void tile_products(const f32x2 (&s)[VerifyTile<K>::RPT][8],
                                              const float* kt_s, const float* qt_s, float* pq_s,
                                              int w, int SV, int row0, int warp, int l, int lr) {
  using Tile = VerifyTile<K>;
  constexpr int LPR = Tile::LPR, RPW = Tile::RPW, RPT = Tile::RPT;
  constexpr int NV = 2 * RPT;                       // values per lane
  constexpr int NSTEP = LPR < NV ? LPR : NV;        // lanes the halving spans
  constexpr int NR = NV / NSTEP;                    // values left per lane
  constexpr int DUP = LPR / NSTEP - 1;              // lane bits holding copies
  const int base = LaneHalveIndex<LPR / 2, NV>::run(l);
  const bool writer = (l & DUP) == 0;
  int wofs[NR];  // the lane's values' offsets in pq_s for token 0
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int v = base + i, g = v >> 1, which = v & 1;
    wofs[i] = which * SV + row0 + (g * Tile::WARPS + warp) * RPW + lr;
  }
  auto token = [&](int t) {
    f32x2 kk[8], qq[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const ulonglong2 k4 = *reinterpret_cast<const ulonglong2*>(kt_s + t * K + 4 * (l + LPR * m));
      const ulonglong2 q4 = *reinterpret_cast<const ulonglong2*>(qt_s + t * K + 4 * (l + LPR * m));
      kk[2 * m] = k4.x; kk[2 * m + 1] = k4.y;
      qq[2 * m] = q4.x; qq[2 * m + 1] = q4.y;
    }
    float x[NV];
#pragma unroll
    for (int g = 0; g < RPT; ++g) {
      // pair accumulators over pairs 0-3 and 4-7, combined pairwise, then
      // the two lanes of the pair
      f32x2 da = mul2(s[g][0], kk[0]), db = mul2(s[g][4], kk[4]);
      f32x2 oa = mul2(s[g][0], qq[0]), ob = mul2(s[g][4], qq[4]);
#pragma unroll
      for (int j = 1; j < 4; ++j) {
        da = fma2(s[g][j], kk[j], da);
        db = fma2(s[g][4 + j], kk[4 + j], db);
        oa = fma2(s[g][j], qq[j], oa);
        ob = fma2(s[g][4 + j], qq[4 + j], ob);
      }
      const float2 dd = unpack2(add2(da, db)), oo = unpack2(add2(oa, ob));
      x[2 * g] = __fadd_rn(dd.x, dd.y);
      x[2 * g + 1] = __fadd_rn(oo.x, oo.y);
    }
    int ignored = 0;  // the same index as `base`
    LaneHalve<LPR / 2, NV>::run(x, l, ignored);
    if (writer) {
#pragma unroll
      for (int i = 0; i < NR; ++i) pq_s[2 * t * SV + wofs[i]] = x[i];
    }
  };
  if constexpr (WC > 0) {
#pragma unroll 2
    for (int t = 0; t < WC; ++t)
      if (t < w) token(t);
  } else {
#pragma unroll 1
    for (int t = 0; t < w; ++t) token(t);
  }
}

// One CTA runs NS consecutive tiles of one (request row, value head): the
// window's side is staged once for all of them, each tile's products with
// it are formed in turn, then each row's u_t and o_t.
template <int K, typename QKV, typename ST, bool NATIVE, bool FULL, int NS, bool KDA, int WC>
__global__ void __launch_bounds__(VerifyTile<K>::THREADS,
                                  VerifyTile<K>::template min_ctas<NATIVE, ST, KDA>())
    gdn_verify_kernel(const VerifyParams p) {
  using Tile = VerifyTile<K>;
  constexpr int LPR = Tile::LPR, RPT = Tile::RPT, VT = Tile::VT;
  constexpr bool BULK = NS > 1;  // tiles arrive by bulk copies into shared memory
  static_assert(!BULK || FULL, "bulk-copied tiles are whole tiles");
  static_assert(!NATIVE || NS == 1, "the native form runs one tile per CTA");
  extern __shared__ __align__(16) unsigned char smem_raw[];

  // launched as a programmatic dependent of the previous kernel in the
  // stream: nothing is read before that kernel has completed and its
  // writes are visible (only the launch itself overlaps its tail)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int span = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile0 = span * NS;  // first tile of this CTA

  // ---- row plan: identical checks in every CTA of the row.  The row's
  // ---- scalars are requested together, not one after another.
  const int32_t* trow = p.slot_table + (size_t)r * p.table_stride;
  const RowScalars rs = row_scalars(p.window_len, trow, p.seq_pos, p.block_size, r);
  const long long t0_raw = p.token_start[r];
  const int w = rs.w;
  SourceSlot src = source_slot(rs, p.W, trow, p.table_stride, p.block_size, p.num_slots);
  long long t0 = 0;
  if (!src.err && src.slot >= 0) {
    t0 = t0_raw;
    if (t0 < 0 || t0 + w > p.num_tokens) src.err = GDN_ROW_ERR_TOKENS;
  }
  if (src.err) {
    if (p.err && tid == 0 && span == 0 && h == 0) atomicOr(p.err, src.err);
    // the reject marker tells the commit not to fold this row's stale record
    if (!NATIVE && tid == 0 && span == 0)
      p.rec_g[((size_t)r * p.HV + h) * p.W * (KDA ? K : 1)] = kRejectedGate;
    return;
  }
  if (src.slot < 0) return;  // null row or empty window: writes nothing

  const int hk = h / (p.HV / p.HK);
  const int l = lane % LPR;   // column lane inside the row group
  const int lr = lane / LPR;  // row inside the warp's row group

  // ---- the first tile's checkpoint loads go out first; they stay in flight
  // ---- while the window is staged.  Row group g holds columns
  // ---- 4*(l + LPR*m) + {0..3}: s[g][2m] = +0,+1 and s[g][2m+1] = +2,+3.
  const ST* S0 = static_cast<const ST*>(p.pool) + ((size_t)src.slot * p.HV + h) * (size_t)p.V * K;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw);
  ST* tbuf = reinterpret_cast<ST*>(smem_raw + kBarBytes);
  const VerifySmem<K, ST, KDA, NATIVE> lay(p.W, NS);
  constexpr uint32_t kTileBytes = BULK ? (uint32_t)(VT * K * sizeof(ST)) : 0u;
  f32x2 s[RPT][8];
  if constexpr (BULK) {
    // one thread requests the first tile as a single bulk copy
    if (tid == 0) {
      mbar_init(bar, 1);
      mbar_expect_tx(bar, kTileBytes);
      bulk_load(tbuf, S0 + (size_t)tile0 * VT * K, kTileBytes, bar);
    }
  } else {
    load_tile<K, ST, FULL>(s, S0, tile0, p.V, warp, l, lr);
  }

  // ---- stage the window: normalised keys and queries, gates, values.
  // ---- Every global load of the stage is issued before any of its
  // ---- arithmetic or shared-memory stores, so the stage costs one memory
  // ---- round trip after the row plan's instead of one per loop pass.
  constexpr int SV = NS * VT;  // staged value rows
  float* sm = reinterpret_cast<float*>(smem_raw + kBarBytes + kTileBytes);
  float* kh_s = sm + lay.kh();
  float* qh_s = sm + lay.qh();
  float* kt_s = sm + lay.kt();
  float* qt_s = sm + lay.qt();
  float* v_s = sm + lay.v();
  float* pq_s = sm + lay.pq();
  float* u_s = sm + lay.u();
  float* gs_s = sm + lay.gs();
  float* ab_s = sm + lay.ab();
  float* al_s = sm + lay.al();
  const QKV* qb = static_cast<const QKV*>(p.q);
  const QKV* kb = static_cast<const QKV*>(p.k);
  const QKV* vb = static_cast<const QKV*>(p.v);

  // value rows as 16-byte pieces when whole tiles and 16-byte aligned rows
  // allow it: piece c covers values [VE c, VE c + VE) of v_s ([W][SV])
  constexpr int VE = 16 / sizeof(QKV);  // values per piece
  constexpr int VPT = SV / VE;          // pieces per token
  const int vpieces = w * VPT;
  const bool vvec = FULL && (reinterpret_cast<uintptr_t>(vb) & 15) == 0 &&
                    ((size_t)p.v_stride * sizeof(QKV)) % 16 == 0;
  const QKV* vrow0 = vb + t0 * p.v_stride + (size_t)h * p.V + (size_t)tile0 * VT;
  auto v_piece = [&](int c) {
    return *reinterpret_cast<const uint4*>(vrow0 + (long long)(c / VPT) * p.v_stride + (c % VPT) * VE);
  };
  uint4 vr[2] = {};
  if (vvec) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (tid + j * Tile::THREADS < vpieces) vr[j] = v_piece(tid + j * Tile::THREADS);
  }
  // gate inputs of the whole window: one lane per token in the last warp
  const bool glane = warp == Tile::WARPS - 1 && lane < w;
  float g_a = 0.f, g_b = 0.f, g_Alog = 0.f, g_dt = 0.f;
  if (glane) {
    const size_t gi = (size_t)(t0 + lane) * p.HV + h;
    if constexpr (!KDA) {
      g_a = p.a[gi];
      g_Alog = p.A_log[h];
      g_dt = p.dt_bias[h];
    }
    g_b = p.b[gi];
  }
  // per-channel decay inputs (KDA): a [T][HV][K], dt_bias [HV][K], four
  // channels per thread and pass when both are 16-byte aligned
  const int kpieces = w * (K / 4);
  const bool kvec = KDA && ((reinterpret_cast<uintptr_t>(p.a) | reinterpret_cast<uintptr_t>(p.dt_bias)) & 15) == 0;
  auto decay_in = [&](int c, float4& av, float4& dv) {
    const int t = c / (K / 4), j = 4 * (c % (K / 4));
    av = *reinterpret_cast<const float4*>(p.a + ((size_t)(t0 + t) * p.HV + h) * K + j);
    dv = *reinterpret_cast<const float4*>(p.dt_bias + (size_t)h * K + j);
  };
  float4 ka = {}, kd = {};
  float kAlog = 0.f;
  if constexpr (KDA) {
    kAlog = p.A_log[h];
    if (kvec && tid < kpieces) decay_in(tid, ka, kd);
  }

  // keys and queries: two tokens per warp and pass (eight per CTA)
  for (int tb = 0; tb < w; tb += 2 * Tile::WARPS) {
    float kx[2][4], qx[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int t = tb + warp + j * Tile::WARPS;
#pragma unroll
      for (int e = 0; e < 4; ++e) kx[j][e] = qx[j][e] = 0.f;
      if (t < w && lane < K / 4) {
        load4(kb + (t0 + t) * p.k_stride + (size_t)hk * K + 4 * lane, kx[j]);
        load4(qb + (t0 + t) * p.q_stride + (size_t)hk * K + 4 * lane, qx[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int t = tb + warp + j * Tile::WARPS;
      if (t >= w) break;  // warp-uniform
      normalise_token<K>(kx[j], qx[j], kh_s + t * K, qh_s + t * K, lane);
    }
  }
  // gates: [W][4] = alpha, beta, -, -
  if (glane) {
    if constexpr (!KDA) gs_s[4 * lane] = gate_decay(g_a, g_Alog, g_dt);
    gs_s[4 * lane + 1] = gate_beta(g_b);
  }
  if constexpr (KDA) {
    const float A = expf(kAlog);  // once per head, not per channel
    if (kvec) {
      auto put = [&](int c, const float4& av, const float4& dv) {
        *reinterpret_cast<float4*>(al_s + 4 * c) =
            make_float4(gate_decay_scaled(av.x, A, dv.x), gate_decay_scaled(av.y, A, dv.y),
                        gate_decay_scaled(av.z, A, dv.z), gate_decay_scaled(av.w, A, dv.w));
      };
      if (tid < kpieces) put(tid, ka, kd);
      for (int c = tid + Tile::THREADS; c < kpieces; c += Tile::THREADS) {
        float4 av, dv;
        decay_in(c, av, dv);
        put(c, av, dv);
      }
    } else {
      for (int i = tid; i < w * K; i += Tile::THREADS) {
        const int t = i / K, j = i % K;
        al_s[i] = gate_decay_scaled(p.a[((size_t)(t0 + t) * p.HV + h) * K + j], A,
                                    p.dt_bias[(size_t)h * K + j]);
      }
    }
  }
  // the value rows of this CTA's tiles, every token
  if (vvec) {
    auto put = [&](int c, const uint4& x) {
      float f[VE];
      widen16(x, f);
#pragma unroll
      for (int e = 0; e < VE; e += 4)
        *reinterpret_cast<float4*>(v_s + VE * c + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
    };
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (tid + j * Tile::THREADS < vpieces) put(tid + j * Tile::THREADS, vr[j]);
    for (int c = tid + 2 * Tile::THREADS; c < vpieces; c += Tile::THREADS) put(c, v_piece(c));
  } else {
    for (int i = tid; i < w * SV; i += Tile::THREADS) {
      const int t = i / SV, row = tile0 * VT + i % SV;
      v_s[i] = (FULL || row < p.V) ? load1(vb + (t0 + t) * p.v_stride + (size_t)h * p.V + row) : 0.f;
    }
  }
  __syncthreads();

  // ---- the window's side: kt, qt, A and B
  float* A_s = ab_s;
  float* B_s = ab_s + p.W * p.W;
  window_side<K, KDA>(w, p.W, kh_s, qh_s, gs_s, al_s, kt_s, qt_s, A_s, B_s, tid, Tile::THREADS,
                      warp, Tile::WARPS, lane);
  __syncthreads();

  const size_t rec_base = ((size_t)r * p.HV + h) * p.W;  // record position 0
  if (!NATIVE && span == 0) {
    // records are 16-byte aligned and K is a multiple of 4
    for (int i = tid; i < w * K / 4; i += Tile::THREADS)
      reinterpret_cast<float4*>(p.rec_k + rec_base * K)[i] = reinterpret_cast<const float4*>(kh_s)[i];
    if constexpr (KDA) {
      for (int i = tid; i < w * K / 4; i += Tile::THREADS)
        reinterpret_cast<float4*>(p.rec_g + rec_base * K)[i] = reinterpret_cast<const float4*>(al_s)[i];
    } else {
      if (tid < w) p.rec_g[rec_base + tid] = gs_s[4 * tid];
    }
  }
  // the products below overwrite khat and qhat in the verify: with bulk
  // copies the tile loop's first barrier orders them after these reads
  if constexpr (!NATIVE && !BULK) __syncthreads();

  // ---- the tiles one after another: C kt_t and C qt_t of every row.  With
  // ---- bulk copies, tile i + 1 is requested into the (single) shared
  // ---- buffer as soon as every warp has moved tile i into registers.
#pragma unroll 1
  for (int i = 0; i < NS; ++i) {
    if constexpr (BULK) {
      const bool ok = mbar_wait(bar, i & 1);
      if (ok) load_tile_shared<K>(s, tbuf, warp, l, lr);
      if (__syncthreads_or(!ok)) {
        // never expected: report, let the copy in flight land, and stop
        if (tid == 0 && p.err) atomicOr(p.err, GDN_ROW_ERR_TIMEOUT);
        mbar_wait(bar, i & 1);
        return;
      }
      if (tid == 0 && i + 1 < NS) {
        fence_proxy_async_shared();
        mbar_expect_tx(bar, kTileBytes);
        bulk_load(tbuf, S0 + (size_t)(tile0 + i + 1) * VT * K, kTileBytes, bar);
      }
    } else {
      if (i > 0) load_tile<K, ST, FULL>(s, S0, tile0 + i, p.V, warp, l, lr);
    }
    tile_products<K, WC>(s, kt_s, qt_s, pq_s, w, SV, i * VT, warp, l, lr);
  }
  __syncthreads();

  // ---- u_t and o_t, one thread per row: d = C kt + sum_{j<t} A u_j,
  // ---- u = beta (v - d), o = C qt + sum_{j<=t} B u_j
  for (int row = tid; row < SV; row += Tile::THREADS) {
    const int hrow = tile0 * VT + row;  // row of the head
    if (!FULL && hrow >= p.V) continue;
    row_recurrence<WC>(row, w, p.W, SV, pq_s, u_s, gs_s, A_s, B_s,
                   [&](int t) { return v_s[t * SV + row]; },
                   p.out + t0 * p.out_stride + (size_t)h * p.V + hrow, p.out_stride,
                   NATIVE ? nullptr : p.rec_u + rec_base * p.V + hrow, p.V);
  }

  // ---- native baseline: fold the tile token by token with the commit's
  // ---- update and write the state after every token
  if constexpr (NATIVE) {
    __syncthreads();
    const size_t snap_step = (size_t)p.HV * p.V * K;
    ST* sbase = static_cast<ST*>(p.snaps) + ((size_t)r * p.W * p.HV + h) * (size_t)p.V * K;
    for (int t = 0; t < w; ++t) {
      f32x2 kk[8], al2[8];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const ulonglong2 k4 = *reinterpret_cast<const ulonglong2*>(kh_s + t * K + 4 * (l + LPR * m));
        kk[2 * m] = k4.x; kk[2 * m + 1] = k4.y;
        if constexpr (KDA) {
          const ulonglong2 a4 = *reinterpret_cast<const ulonglong2*>(al_s + t * K + 4 * (l + LPR * m));
          al2[2 * m] = a4.x; al2[2 * m + 1] = a4.y;
        } else {
          al2[2 * m] = al2[2 * m + 1] = pack2(gs_s[4 * t], gs_s[4 * t]);
        }
      }
#pragma unroll
      for (int g = 0; g < RPT; ++g) {
        const int tr = (g * Tile::WARPS + warp) * Tile::RPW + lr;  // row in the tile
        const int hrow = tile0 * VT + tr;
        const float u = u_s[t * SV + tr];
        const f32x2 u2 = pack2(u, u);
#pragma unroll
        for (int j = 0; j < 8; ++j) s[g][j] = fold2(s[g][j], al2[j], u2, kk[j]);
        if (FULL || hrow < p.V) {
          ST* dst = sbase + t * snap_step + (size_t)hrow * K + 4 * l;
#pragma unroll
          for (int m = 0; m < 4; ++m) store_state_pairs(dst + 4 * LPR * m, s[g][2 * m], s[g][2 * m + 1]);
        }
      }
    }
  }
}

template <int K, typename QKV, typename ST, bool NATIVE, bool FULL, int NS, bool KDA, int WC = 0>
static void launch_tiles(const VerifyParams& p, int ntiles, cudaStream_t stream) {
  using Tile = VerifyTile<K>;
  dim3 grid(ntiles / NS, p.HV, p.batch);
  const size_t smem = VerifySmem<K, ST, KDA, NATIVE>(p.W, NS).bytes(NS);
  auto kern = gdn_verify_kernel<K, QKV, ST, NATIVE, FULL, NS, KDA, WC>;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  // programmatic stream serialization: the CTAs may be launched while the
  // previous kernel's last CTAs run; each waits for it at its first
  // instruction (the launch latency of back-to-back layers overlaps)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Tile::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kern, p);
}

// The verify runs 4 (else 2) tiles of a head per CTA when they divide the
// head (two 64-row tiles for a 128-row head at K = 128); the native
// baseline, and heads smaller than a tile, one per CTA.  A multi-tile CTA
// with a 4- or 6-token record stride (three or five drafted tokens plus the
// last accepted one) runs a build of the kernel with the token loops
// unrolled.
template <int K, typename QKV, typename ST, bool NATIVE, bool KDA>
static int launch_one(const VerifyParams& p, cudaStream_t stream) {
  using Tile = VerifyTile<K>;
  const int ntiles = (p.V + Tile::VT - 1) / Tile::VT;
  const bool full = p.V % Tile::VT == 0;
  bool done = false;
  if constexpr (!NATIVE) {
    if (full && ntiles % 4 == 0) {
      if (p.W == 4) launch_tiles<K, QKV, ST, NATIVE, true, 4, KDA, 4>(p, ntiles, stream);
      else if (p.W == 6) launch_tiles<K, QKV, ST, NATIVE, true, 4, KDA, 6>(p, ntiles, stream);
      else launch_tiles<K, QKV, ST, NATIVE, true, 4, KDA>(p, ntiles, stream);
      done = true;
    } else if (full && ntiles % 2 == 0) {
      if (p.W == 4) launch_tiles<K, QKV, ST, NATIVE, true, 2, KDA, 4>(p, ntiles, stream);
      else if (p.W == 6) launch_tiles<K, QKV, ST, NATIVE, true, 2, KDA, 6>(p, ntiles, stream);
      else launch_tiles<K, QKV, ST, NATIVE, true, 2, KDA>(p, ntiles, stream);
      done = true;
    }
  }
  if (!done) {
    if (full) launch_tiles<K, QKV, ST, NATIVE, true, 1, KDA>(p, ntiles, stream);
    else launch_tiles<K, QKV, ST, NATIVE, false, 1, KDA>(p, ntiles, stream);
  }
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <int K, bool NATIVE, bool KDA>
static int dispatch_dtypes(const VerifyParams& p, int qkv_dtype, int state_dtype,
                           cudaStream_t stream) {
  if (qkv_dtype == GDN_DTYPE_F32 && state_dtype == GDN_DTYPE_F32)
    return launch_one<K, float, float, NATIVE, KDA>(p, stream);
  if (qkv_dtype == GDN_DTYPE_F32 && state_dtype == GDN_DTYPE_BF16)
    return launch_one<K, float, __nv_bfloat16, NATIVE, KDA>(p, stream);
  if (qkv_dtype == GDN_DTYPE_BF16 && state_dtype == GDN_DTYPE_F32)
    return launch_one<K, __nv_bfloat16, float, NATIVE, KDA>(p, stream);
  return launch_one<K, __nv_bfloat16, __nv_bfloat16, NATIVE, KDA>(p, stream);
}

// One head width and gate kind, native or verify, every dtype pair.
template <int K, bool KDA>
static int dispatch_native(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,
                           cudaStream_t stream) {
  return native ? dispatch_dtypes<K, true, KDA>(p, qkv_dtype, state_dtype, stream)
                : dispatch_dtypes<K, false, KDA>(p, qkv_dtype, state_dtype, stream);
}

}  // namespace gdn
