// gdn_verify.cu -- speculative verify and native per-draft snapshot kernels.
//
// One CTA of 4 warps runs the whole draft window over up to four tiles of VT
// state rows (32 for K = 128) of one (request row, value head), one tile
// after another, with the tile held in registers (tokenspeed PR "feat: add
// Qwen3.5 GDN ReplaySSM", Summary and Implementation: a cooperative 4-warp
// CTA per 128x128 state head).  The window's normalised keys and queries,
// gates and values are staged once per CTA for all of its tiles: that
// staging and the row plan cost as many instructions as the recurrence of
// one tile, so a head run as four separate tile CTAs paid them four times.
// Tiles reach the CTA as single bulk copies (cp.async.bulk, one thread, one
// instruction per 16 KiB tile) into one shared-memory buffer, completed
// through an mbarrier: tile i + 1 is requested as soon as every warp has
// moved tile i into registers, so it streams in while tile i runs (80
// registers and six CTAs per SM for an fp32 state, 72 and seven for bf16).
// A CTA with a single tile (the native form) loads it straight into
// registers.  Rows of S are independent given (khat, qhat, alpha, beta,
// v_i), so tiles never communicate; the only reductions are over K, inside
// a group of K/16 lanes, by warp shuffles.
//
// Register layout of a tile, for K = 128: LPR = 8 lanes share one state row
// and each lane holds 16 of its columns, as four 4-column chunks at columns
// 4 * (l + LPR * m), m = 0..3, kept as eight packed fp32 pairs; a warp's
// load of chunk m reads whole 128-byte lines.  A warp covers RPW = 32 / LPR
// rows per row group and each thread keeps RPT row groups.
//
// Per token: H = alpha * S; both dot products are taken in one pass over H,
// d = H khat and H qhat; then u = beta * (v - d), S = H + u khat^T and
// o = S qhat evaluated as H qhat + u * (khat . qhat), the same value in
// exact arithmetic with the output off the state update's critical path.
// The two lane sums share their shuffles: one exchange leaves d on the lower
// half of a row's lanes and o on the upper half, each half then sums its own
// value, and d is broadcast back (4 shuffles per row and token, not 6).
// With the per-channel (KDA) decay, H = S diag(alpha_t): the staging computes
// one gate per (token, channel), and each thread scales its own columns by
// their gates before the token's keys and queries are loaded.
//
// VERIFY mode writes o_t and the replay record (u_t, khat_t, alpha_t) and no
// state (vLLM PR "[Spec Decode][Qwen4Exp] RecoverSSM for Qwen GDN and the
// PLE short conv", Purpose).  NATIVE mode writes o_t and the full state after
// every token instead, one tile per CTA.  Both run the identical per-token
// arithmetic on every row, so their outputs agree bit for bit however the
// tiles are grouped into CTAs, and the state update is the commit's fold
// (which VERIFY mode skips after the window's last token: that state is
// never read).
#include <type_traits>

#include "gdn_async.cuh"
#include "gdn_device.cuh"
#include "gdn_launch.h"

namespace gdn {

template <int K>
struct VerifyTile {
  static constexpr int LPR = K / 16;              // lanes per state row
  static constexpr int RPW = 32 / LPR;            // rows per warp per row group
  static constexpr int RPT = (K == 128) ? 2 : 1;  // row groups per thread
  static constexpr int WARPS = 4;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int VT = WARPS * RPW * RPT;    // state rows per tile
  // CTAs per SM the registers must allow, as measured: seven (72 registers)
  // for the native form and for the verify with a bf16 state; six (80
  // registers) for the verify with an fp32 state, which spills at 72.  The
  // per-channel (KDA) decay is applied before a token's keys and queries are
  // loaded, so its gate registers are free again and it keeps the same
  // budgets.
  template <bool NATIVE, typename ST, bool KDA>
  static constexpr int min_ctas() {
    return (!NATIVE && sizeof(ST) == 4) ? 6 : 7;
  }
};

// Dynamic shared memory of one verify CTA covering NS tiles, in bytes: the
// mbarrier (16 bytes), the tile buffer the bulk copies fill (NS > 1 only),
// then the staged keys, queries, values and gates (plus, for the
// per-channel KDA gate, the window's [W][K] decay vectors).
template <int K, typename ST>
__host__ __device__ constexpr size_t verify_tile_bytes(int NS) {
  return NS > 1 ? (size_t)VerifyTile<K>::VT * K * sizeof(ST) : 0;
}
template <int K, typename ST, bool KDA>
__host__ __device__ constexpr size_t verify_smem_bytes(int W, int NS) {
  return 16 + verify_tile_bytes<K, ST>(NS) +
         sizeof(float) * (size_t)W * (2 * K + NS * VerifyTile<K>::VT + 4 + (KDA ? K : 0));
}

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

// The draft window over one tile whose state is in s.  vt_off: this tile's
// first row inside the CTA's staged value rows.  al_s: the window's
// per-channel decay vectors [W][K] (KDA), unused for the scalar gate.
template <int K, typename ST, bool NATIVE, bool FULL, bool KDA>
__device__ __forceinline__ void run_tile(f32x2 (&s)[VerifyTile<K>::RPT][8], const VerifyParams& p,
                                         int tile, int h, int r, int w, long long t0, int vt_off,
                                         int vrow_stride, const float* kh_s, const float* qh_s,
                                         const float* v_s, const float* gs_s, const float* al_s,
                                         int warp, int l, int lr) {
  using Tile = VerifyTile<K>;
  constexpr int LPR = Tile::LPR, RPW = Tile::RPW, RPT = Tile::RPT, VT = Tile::VT;
  const size_t rec_base = ((size_t)r * p.HV + h) * p.W;
  // the d half (lower LPR/2 lanes) and the o half of a row's lanes after
  // the first exchange; the first o lane writes the row's outputs
  const bool upper = LPR > 1 && (l & (LPR / 2)) != 0;
  const int lane = lr * LPR + l;
  const bool writer = (l == LPR / 2);
  int rows[RPT];
  float* optr[RPT];
  float* uptr[RPT];
  ST* sptr[RPT];
#pragma unroll
  for (int g = 0; g < RPT; ++g) {
    rows[g] = tile * VT + (g * Tile::WARPS + warp) * RPW + lr;
    optr[g] = p.out + t0 * p.out_stride + (size_t)h * p.V + rows[g];
    uptr[g] = NATIVE ? nullptr : p.rec_u + rec_base * p.V + rows[g];
    sptr[g] = NATIVE ? static_cast<ST*>(p.snaps) + ((size_t)r * p.W * p.HV + h) * (size_t)p.V * K +
                           (size_t)rows[g] * K + 4 * l
                     : nullptr;
  }
  const size_t snap_step = (size_t)p.HV * p.V * K;
  // ---- the draft window, token by token, state in registers.  In VERIFY
  // ---- mode the state after the last token is never read: that token runs
  // ---- without the update.
  auto token = [&](int t, auto update_tag) {
    constexpr bool UPDATE = decltype(update_tag)::value;
    const ulonglong2 gq = *reinterpret_cast<const ulonglong2*>(gs_s + 4 * t);
    [[maybe_unused]] const f32x2 al2 = gq.x;  // (alpha, alpha); unused with the KDA decay
    const float2 bk = unpack2(gq.y);
    const float be = bk.x, kq = bk.y;
    if constexpr (KDA) {
      // H = S diag(alpha): each pair of this thread's columns by its own
      // gates, applied before the keys and queries are loaded so that the
      // gate registers are free again
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const ulonglong2 a4 = *reinterpret_cast<const ulonglong2*>(al_s + t * K + 4 * (l + LPR * m));
#pragma unroll
        for (int g = 0; g < RPT; ++g) {
          s[g][2 * m] = mul2(s[g][2 * m], a4.x);
          s[g][2 * m + 1] = mul2(s[g][2 * m + 1], a4.y);
        }
      }
    }
    f32x2 kk[8], qq[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const ulonglong2 k4 = *reinterpret_cast<const ulonglong2*>(kh_s + t * K + 4 * (l + LPR * m));
      const ulonglong2 q4 = *reinterpret_cast<const ulonglong2*>(qh_s + t * K + 4 * (l + LPR * m));
      kk[2 * m] = k4.x; kk[2 * m + 1] = k4.y;
      qq[2 * m] = q4.x; qq[2 * m + 1] = q4.y;
    }
#pragma unroll
    for (int g = 0; g < RPT; ++g) {
      // H = alpha * S (the per-channel decay was applied above)
      if constexpr (!KDA) {
#pragma unroll
        for (int j = 0; j < 8; ++j) s[g][j] = mul2(s[g][j], al2);
      }
      // d = H khat and H qhat in one pass: pair accumulators over pairs
      // 0-3 and 4-7, combined pairwise, lanes summed, then the LPR lanes
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
      float d = __fadd_rn(dd.x, dd.y), o = __fadd_rn(oo.x, oo.y);
      if (LPR > 1) {
        // halving exchange: the d half keeps d and sends o, the o half the
        // reverse; then each half sums its own value over its lanes
        const float keep = upper ? o : d, send = upper ? d : o;
        float x = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, LPR / 2));
#pragma unroll
        for (int off = LPR / 4; off >= 1; off >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, off));
        d = __shfl_sync(0xffffffffu, x, lane - l);  // every lane takes d from the row's first lane
        o = x;                                      // meaningful on the o half
      }
      const float vi = (FULL || rows[g] < p.V) ? v_s[t * vrow_stride + vt_off + rows[g] - tile * VT] : 0.f;
      const float u = __fmul_rn(be, __fsub_rn(vi, d));
      o = __fmaf_rn(u, kq, o);
      // S = H + u khat^T
      if (UPDATE) {
        const f32x2 u2 = pack2(u, u);
#pragma unroll
        for (int j = 0; j < 8; ++j) s[g][j] = fma2(u2, kk[j], s[g][j]);
      }
      if (FULL || rows[g] < p.V) {
        if (writer) {
          *optr[g] = o;
          if (!NATIVE) *uptr[g] = u;
        }
        if (NATIVE) {
#pragma unroll
          for (int m = 0; m < 4; ++m)
            store_state_pairs(sptr[g] + 4 * LPR * m, s[g][2 * m], s[g][2 * m + 1]);
        }
      }
      optr[g] += p.out_stride;
      if (!NATIVE) uptr[g] += p.V;
      if (NATIVE) sptr[g] += snap_step;
    }
  };
  if constexpr (NATIVE) {
    for (int t = 0; t < w; ++t) token(t, std::true_type{});
  } else {
    for (int t = 0; t + 1 < w; ++t) token(t, std::true_type{});
    token(w - 1, std::false_type{});
  }
}

// One CTA runs NS consecutive tiles of one (request row, value head): the
// window's keys, queries, gates and values are staged once for all of them,
// then each tile's checkpoint rows are loaded and its window run in turn.
template <int K, typename QKV, typename ST, bool NATIVE, bool FULL, int NS, bool KDA>
__global__ void __launch_bounds__(VerifyTile<K>::THREADS,
                                  VerifyTile<K>::template min_ctas<NATIVE, ST, KDA>())
    gdn_verify_kernel(const VerifyParams p) {
  using Tile = VerifyTile<K>;
  constexpr int LPR = Tile::LPR, RPT = Tile::RPT, VT = Tile::VT;
  constexpr bool BULK = NS > 1;  // tiles arrive by bulk copies into shared memory
  static_assert(!BULK || FULL, "bulk-copied tiles are whole tiles");
  extern __shared__ __align__(16) unsigned char smem_raw[];

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
  // ---- while the window's inputs are staged.  Row group g holds columns
  // ---- 4*(l + LPR*m) + {0..3}: s[g][2m] = +0,+1 and s[g][2m+1] = +2,+3.
  const ST* S0 = static_cast<const ST*>(p.pool) + ((size_t)src.slot * p.HV + h) * (size_t)p.V * K;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw);
  ST* tbuf = reinterpret_cast<ST*>(smem_raw + 16);
  constexpr uint32_t kTileBytes = (uint32_t)verify_tile_bytes<K, ST>(NS);
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

  // ---- stage normalised keys / queries, their dot product, the gates and
  // ---- the value rows of all NS tiles for the whole window in shared
  // ---- memory.  Every global load of the stage is issued before any of its
  // ---- arithmetic or shared-memory stores, so the stage costs one memory
  // ---- round trip after the row plan's instead of one per loop pass (a
  // ---- load is not moved above an earlier pass's stores by the compiler).
  constexpr int SV = NS * VT;           // staged value rows
  float* kh_s = reinterpret_cast<float*>(smem_raw + 16 + kTileBytes);  // [W][K]
  float* qh_s = kh_s + p.W * K;         // [W][K]
  float* v_s = qh_s + p.W * K;          // [W][SV]
  float* gs_s = v_s + p.W * SV;         // [W][4]: alpha, alpha, beta, khat . qhat
  float* al_s = gs_s + 4 * p.W;         // [W][K]: per-channel decay (KDA only)
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
      float ks = __fmul_rn(kx[j][0], kx[j][0]), qs = __fmul_rn(qx[j][0], qx[j][0]);
#pragma unroll
      for (int e = 1; e < 4; ++e) {
        ks = __fmaf_rn(kx[j][e], kx[j][e], ks);
        qs = __fmaf_rn(qx[j][e], qx[j][e], qs);
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        ks = __fadd_rn(ks, __shfl_xor_sync(0xffffffffu, ks, off));
        qs = __fadd_rn(qs, __shfl_xor_sync(0xffffffffu, qs, off));
      }
      // x / sqrt(|x|^2 + eps) as x * rsqrt(|x|^2 + eps), rsqrt correctly rounded
      const float kr = __frsqrt_rn(__fadd_rn(ks, kL2NormEps));
      const float qr = __frsqrt_rn(__fadd_rn(qs, kL2NormEps));
      float kn[4], qn[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kn[e] = __fmul_rn(kx[j][e], kr);
        qn[e] = __fmul_rn(qx[j][e], qr);
      }
      float kq = __fmul_rn(kn[0], qn[0]);
#pragma unroll
      for (int e = 1; e < 4; ++e) kq = __fmaf_rn(kn[e], qn[e], kq);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) kq = __fadd_rn(kq, __shfl_xor_sync(0xffffffffu, kq, off));
      if (lane < K / 4) {
        *reinterpret_cast<float4*>(kh_s + t * K + 4 * lane) = make_float4(kn[0], kn[1], kn[2], kn[3]);
        *reinterpret_cast<float4*>(qh_s + t * K + 4 * lane) = make_float4(qn[0], qn[1], qn[2], qn[3]);
      }
      if (lane == 0) gs_s[4 * t + 3] = kq;
    }
  }
  // gates
  if (glane) {
    if constexpr (!KDA) {
      const float al = gate_decay(g_a, g_Alog, g_dt);
      gs_s[4 * lane] = al;
      gs_s[4 * lane + 1] = al;
    }
    gs_s[4 * lane + 2] = gate_beta(g_b);
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

  // ---- the tiles one after another.  With bulk copies, tile i + 1 is
  // ---- requested into the (single) shared buffer as soon as every warp has
  // ---- moved tile i into registers, so it streams in while tile i runs.
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
    run_tile<K, ST, NATIVE, FULL, KDA>(s, p, tile0 + i, h, r, w, t0, i * VT, SV, kh_s, qh_s, v_s,
                                       gs_s, al_s, warp, l, lr);
  }
}

template <int K, typename QKV, typename ST, bool NATIVE, bool FULL, int NS, bool KDA>
static void launch_tiles(const VerifyParams& p, int ntiles, cudaStream_t stream) {
  using Tile = VerifyTile<K>;
  dim3 grid(ntiles / NS, p.HV, p.batch);
  const size_t smem = verify_smem_bytes<K, ST, KDA>(p.W, NS);
  auto kern = gdn_verify_kernel<K, QKV, ST, NATIVE, FULL, NS, KDA>;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  kern<<<grid, Tile::THREADS, smem, stream>>>(p);
}

// The verify runs 4 (else 2) tiles of a head per CTA when they divide the
// head; the native baseline, and heads smaller than a tile, one per CTA.
template <int K, typename QKV, typename ST, bool NATIVE, bool KDA>
static int launch_one(const VerifyParams& p, cudaStream_t stream) {
  using Tile = VerifyTile<K>;
  const int ntiles = (p.V + Tile::VT - 1) / Tile::VT;
  const bool full = p.V % Tile::VT == 0;
  bool done = false;
  if constexpr (!NATIVE) {
    if (full && ntiles % 4 == 0) {
      launch_tiles<K, QKV, ST, NATIVE, true, 4, KDA>(p, ntiles, stream);
      done = true;
    } else if (full && ntiles % 2 == 0) {
      launch_tiles<K, QKV, ST, NATIVE, true, 2, KDA>(p, ntiles, stream);
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

template <int K>
static int dispatch_modes(const VerifyParams& p, int qkv_dtype, int state_dtype, bool native,
                          bool kda, cudaStream_t stream) {
  if (kda)
    return native ? dispatch_dtypes<K, true, true>(p, qkv_dtype, state_dtype, stream)
                  : dispatch_dtypes<K, false, true>(p, qkv_dtype, state_dtype, stream);
  return native ? dispatch_dtypes<K, true, false>(p, qkv_dtype, state_dtype, stream)
                : dispatch_dtypes<K, false, false>(p, qkv_dtype, state_dtype, stream);
}

int launch_verify(const VerifyParams& p, int head_k, int qkv_dtype, int state_dtype,
                  bool native, bool kda, cudaStream_t stream) {
  switch (head_k) {
    case 16: return dispatch_modes<16>(p, qkv_dtype, state_dtype, native, kda, stream);
    case 32: return dispatch_modes<32>(p, qkv_dtype, state_dtype, native, kda, stream);
    case 64: return dispatch_modes<64>(p, qkv_dtype, state_dtype, native, kda, stream);
    case 128: return dispatch_modes<128>(p, qkv_dtype, state_dtype, native, kda, stream);
    default: return GDN_ERR_UNSUPPORTED;
  }
}

}  // namespace gdn
