// State walks of the γ and θ gradients on the tensor cores (tcgen05, TMEM,
// TMA).
//
// The γ/θ gradients (ret_chunkwise_param_grads) need the states at the
// chunk boundaries, S_c (after chunk c, from S_in) and dS_c (their
// gradients, from dS_out), and the weighted products of the two:
//   S_c      = γ^{b_c} S_{c−1} + Σ_{i∈c} kf_iᵀ v_i,     kf_i = d_k^{-1/2} γ^{b_c−1−j} R(i) k_i
//   dS_{c−1} = γ^{b_c} dS_c   + Σ_{i∈c} qb_iᵀ dO_i,    qb_i = γ^{j+1} R(i) q_i
//   γ·dγ ∋ Σ_c w_c <S_c, dS_c>,   dθ_p ∋ Σ_c u_c Σ_v (S_c[2p+1,v] dS_c[2p,v] − S_c[2p,v] dS_c[2p+1,v])
// (j the row inside the chunk; the walk weights w_c, u_c are the ones of the
// fp32 walks in kernels_grad.cuh).  Each chunk's update is a dense
// contraction over its 128 rows, so it runs on the tensor cores: the
// transposed update ΔSᵀ [v × k] = Vᵀ · kf (A = the bf16 value rows, exact,
// MN-major; B = kf, MN-major).  kf and qb are not bf16 numbers (rotation and
// decay weights), so each is stored as two bf16 parts hi + lo (hi = bf16(x),
// lo = bf16(x − hi): 16 significant bits) and the update takes two MMAs into
// one fp32 accumulator; the fp32 state itself lives in the drain warps'
// registers, as in the chunk kernels.
//
// CTA = (128-column v tile, 128-column k tile, b·h); block = 576 threads:
// warp 0 TMA producer, warp 1 MMA issuer, warps 2..17 drain warps (drain
// warp w reads TMEM lanes 32·(warp % 4) … +31 and k columns 32·(w / 4) …
// +31).  Two shared-memory stages of (value rows, kf hi, kf lo) = 96 KB each
// and two 128-column accumulators in TMEM, so the loads of the next chunk
// and its MMAs overlap the drain of the current one.
//   FWD: chunks in order; S_c stored per chunk ([BH][C][d_k][d_v] fp32).
//   !FWD: chunks from the last; after each chunk the products of dS_{c−1}
//   with the stored S_{c−1} (S_in for c = 0); the weighted sums go out per
//   64 × 64 sub-tile, in the layout of the fp32 walks' partials.
#pragma once

#include "common.cuh"
#include "tc_primitives.cuh"

namespace ret {
namespace tcw {

using namespace ret::tc;

constexpr int CH = 128;                        // chunk rows
constexpr int VT = 128;                        // v columns per CTA
constexpr int KT = 128;                        // k columns per CTA
constexpr int NCW = 16;                        // drain warps
constexpr int NTHREADS = (NCW + 2) * 32;
constexpr int NST = 2;                         // shared-memory stages
constexpr int SPT = KT / 4;                    // state values per drain thread
constexpr uint32_t BOX = CH * 64 * 2;          // 64 columns × 128 rows, bf16 (16 KB)
constexpr uint32_t TILE = 2 * BOX;             // 128 columns
constexpr uint32_t STAGE = 3 * TILE;           // value rows, kf hi, kf lo
enum Bar : int { FULL0 = 0, EMPTY0 = FULL0 + NST, DFULL0 = EMPTY0 + NST, DFREE0 = DFULL0 + 2,
                 DONE = DFREE0 + 2, NBAR_ };
constexpr uint32_t OFF_BAR = NST * STAGE;
constexpr uint32_t OFF_TPTR = OFF_BAR + NBAR_ * 8;
constexpr uint32_t OFF_RED = (OFF_TPTR + 16 + 7) & ~7u;   // [4 k ranges][4 quarters][17] doubles
constexpr uint32_t USED = OFF_RED + 4 * 4 * 17 * 8;
constexpr uint32_t SMEM_BYTES = USED + 1024;               // slack for 1024-byte alignment
constexpr uint32_t T_COLS = 2 * KT;                        // two accumulators
constexpr float kKappa = 0.5f * (CH - 1);

struct WalkTcArgs {
  const float* s0;      // FWD: S_in; !FWD: dS_out ([BH][d_k][d_v] fp32), or null (zero)
  const float* s_in;    // !FWD: S_in (the state before chunk 0), or null
  float* states;        // [BH][C][d_k][d_v]: written (FWD), read (!FWD)
  double* gpart;        // !FWD: [BH][(d_k/64)·(d_v/64)] weighted Σ <S_c, dS_c> per 64 × 64 sub-tile
  float* zpart;         // !FWD: [BH][(d_k/64)·(d_v/64)][32] weighted Σ Z_c per pair of the sub-tile
  int H, L, Lp, d_k, d_v, C;
  float pos0;
};

// tm_b: the value rows (v or dO) [BH][L][d_v], boxes 64 × 128 × 1;
// tm_hi / tm_lo: the parts of kf or qb [BH·Lp][d_k], boxes 64 × 128.
template <bool FWD>
__global__ void __launch_bounds__(NTHREADS, 1)
    walk_tc_kernel(const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_hi,
                   const __grid_constant__ CUtensorMap tm_lo, WalkTcArgs a, CallConsts cc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8u * static_cast<uint32_t>(i); };
  auto stage = [&](int s) -> uint32_t { return sb + static_cast<uint32_t>(s) * STAGE; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v0 = blockIdx.x * VT, k0 = blockIdx.y * KT;
  const int bh = blockIdx.z;
  const int h = bh % a.H;
  const int C = a.C;
  const int rl = a.L - (C - 1) * CH;   // rows of the last chunk
  auto cix = [&](int i) -> int { return FWD ? i : C - 1 - i; };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_hi);
    tma_prefetch_desc(&tm_lo);
    for (int i = 0; i < NBAR_; ++i) mbar_init(bar(i), (i == DFREE0 || i == DFREE0 + 1) ? NCW : 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + OFF_TPTR, T_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TPTR);
  double* red = reinterpret_cast<double*>(smem + OFF_RED);

  if (warp == 0) {
    // ------------------------------ TMA producer ---------------------------
    if (lane == 0) {
      int issued = -1;
      for (int i = 0; i < C; ++i) {
        const int s = i % NST, c = cix(i);
        if (i >= NST && !mbar_wait(bar(EMPTY0 + s), static_cast<uint32_t>((i - NST) / NST) & 1u, 0x601)) break;
        mbar_arrive_expect_tx(bar(FULL0 + s), STAGE);
        const uint32_t st = stage(s);
        const int y = bh * a.Lp + c * CH;
        for (int b = 0; b < 2; ++b) {
          tma_load_3d(st + b * BOX, &tm_b, v0 + 64 * b, c * CH, bh, bar(FULL0 + s));
          tma_load_2d(st + TILE + b * BOX, &tm_hi, k0 + 64 * b, y, bar(FULL0 + s));
          tma_load_2d(st + 2 * TILE + b * BOX, &tm_lo, k0 + 64 * b, y, bar(FULL0 + s));
        }
        issued = i;
      }
      // never leave with copies still landing
      if (status_aborted())
        for (int i = issued > 0 ? issued - 1 : 0; i <= issued; ++i)
          mbar_wait(bar(FULL0 + i % NST), static_cast<uint32_t>(i / NST) & 1u, 0x6f1, kWaitBudgetCycles / 8);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer -----------------------------
    if (lane == 0) {
      constexpr uint32_t ID = idesc_bf16_f32(128, KT, 1, 1);   // both operands MN-major
      for (int i = 0; i < C; ++i) {
        const int s = i % NST, d = i & 1;
        if (!mbar_wait(bar(FULL0 + s), static_cast<uint32_t>(i / NST) & 1u, 0x611)) break;
        if (i >= 2 && !mbar_wait(bar(DFREE0 + d), static_cast<uint32_t>((i - 2) >> 1) & 1u, 0x612)) break;
        tc_fence_after();
        const uint32_t st = stage(s);
        const uint64_t dB = sdesc_sw128(st, BOX, 1024);
        const uint64_t dHi = sdesc_sw128(st + TILE, BOX, 1024);
        const uint64_t dLo = sdesc_sw128(st + 2 * TILE, BOX, 1024);
        const uint32_t tD = tmem + static_cast<uint32_t>(d * KT);
#pragma unroll
        for (int k = 0; k < CH / 16; ++k)   // +2048 bytes (16 rows) per step
          mma_ss(tD, dB + static_cast<uint64_t>(k * 128), dHi + static_cast<uint64_t>(k * 128), ID,
                 k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < CH / 16; ++k)
          mma_ss(tD, dB + static_cast<uint64_t>(k * 128), dLo + static_cast<uint64_t>(k * 128), ID, 1u);
        mma_commit(bar(DFULL0 + d));
        mma_commit(bar(EMPTY0 + s));
      }
      // all issued MMAs finish before TMEM is released
      mma_commit(bar(DONE));
      mbar_wait(bar(DONE), 0, 0x6ff);
    }
  } else {
    // ------------------------------ drain warps ----------------------------
    const int w = warp - 2;                   // 0..15
    const int quarter = warp & 3;             // TMEM lanes 32·quarter … +31
    const int kr = w >> 2;                    // k columns 32·kr … +31 of the tile
    const int vl = 32 * quarter + lane;       // local v
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    const int v = v0 + vl, kb = k0 + kr * SPT;
    const bool vlive = v < a.d_v;             // always true: d_v is a multiple of 128
    const size_t plane = static_cast<size_t>(a.d_k) * a.d_v;
    auto at = [&](int u) -> size_t { return static_cast<size_t>(kb + u) * a.d_v + v; };
    const float lg = cc.lg2g[h];

    float S[SPT];
#pragma unroll
    for (int u = 0; u < SPT; ++u) S[u] = (a.s0 && vlive) ? a.s0[static_cast<size_t>(bh) * plane + at(u)] : 0.f;

    // !FWD: weighted boundary products of S (= dS_c) with S_c.  The pair
    // terms are summed over the warp's 32 v lanes at every boundary (a
    // halving exchange: after it lanes 2p and 2p + 1 hold pair p), so each
    // lane keeps one running sum.
    double gacc = 0.0, zacc = 0.0;
    auto boundary = [&](int c) {
      const float* src = c >= 0 ? a.states + (static_cast<size_t>(bh) * C + c) * plane
                                : (a.s_in ? a.s_in + static_cast<size_t>(bh) * plane : nullptr);
      float ip = 0.f, z[SPT / 2];
#pragma unroll
      for (int p = 0; p < SPT / 2; ++p) {
        const float s0v = src ? src[at(2 * p)] : 0.f, s1v = src ? src[at(2 * p + 1)] : 0.f;
        ip = fmaf(s0v, S[2 * p], fmaf(s1v, S[2 * p + 1], ip));
        z[p] = fmaf(s1v, S[2 * p], -(s0v * S[2 * p + 1]));
      }
#pragma unroll
      for (int n = SPT / 4, o = 16; n >= 1; n >>= 1, o >>= 1) {   // 16 pairs → 1 per lane
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int p = 0; p < n; ++p) {
          const float keep = up ? z[p + n] : z[p], send = up ? z[p] : z[p + n];
          z[p] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      const float zs = z[0] + __shfl_xor_sync(0xffffffffu, z[0], 1);
      float wg, wt;
      if (c == C - 1) {
        wg = static_cast<float>(rl - 1) - kKappa;
        wt = -(a.pos0 + static_cast<float>((C - 1) * CH) + kKappa);
      } else if (c < 0) {
        wg = 1.f + kKappa;
        wt = a.pos0 + kKappa;
      } else {
        wg = wt = static_cast<float>(CH);
      }
      gacc += static_cast<double>(wg) * ip;
      zacc += static_cast<double>(wt) * zs;
    };
    if (!FWD) boundary(C - 1);

    bool ok = true;
    for (int i = 0; i < C && ok; ++i) {
      const int c = cix(i), d = i & 1;
      if (!mbar_wait(bar(DFULL0 + d), static_cast<uint32_t>(i >> 1) & 1u, 0x621)) { ok = false; break; }
      tc_fence_after();
      uint32_t r0[16], r1[16];
      tmem_ld16(tmem + static_cast<uint32_t>(d * KT) + lane_off + kr * SPT, r0);
      tmem_ld16(tmem + static_cast<uint32_t>(d * KT) + lane_off + kr * SPT + 16, r1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DFREE0 + d));
      const float g = gpow(lg, static_cast<float>(c == C - 1 ? rl : CH));   // γ^{b_c}
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        S[u] = fmaf(g, S[u], __uint_as_float(r0[u]));
        S[16 + u] = fmaf(g, S[16 + u], __uint_as_float(r1[u]));
      }
      if (FWD) {
        float* dst = a.states + (static_cast<size_t>(bh) * C + c) * plane;
#pragma unroll
        for (int u = 0; u < SPT; ++u) dst[at(u)] = S[u];
      } else {
        boundary(c - 1);
      }
    }
    if (!FWD) {
      // sums over this warp's 32 v lanes, then per (k range, quarter) in shared memory
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gacc += __shfl_xor_sync(0xffffffffu, gacc, o);
      double* rr = red + (kr * 4 + quarter) * 17;
      if ((lane & 1) == 0) rr[lane >> 1] = zacc;
      if (lane == 0) rr[16] = gacc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (!FWD && threadIdx.x < 4 * 32) {
    // sub-tile (tk, tv) of 64 × 64 = k ranges 2·(tk%2) … +1, quarters 2·(tv%2) … +1
    const int t = threadIdx.x;   // (sub-tile = t / 32, pair = t % 32)
    const int st = t >> 5, pl = t & 31;
    const int tkl = st >> 1, tvl = st & 1;
    const int kr = 2 * tkl + (pl >> 4), p = pl & 15;
    const int ntv = a.d_v / 64, ntiles = (a.d_k / 64) * ntv;
    const int tk = 2 * blockIdx.y + tkl, tv = 2 * blockIdx.x + tvl;
    const size_t slot = static_cast<size_t>(bh) * ntiles + static_cast<size_t>(tk) * ntv + tv;
    const double z = red[(kr * 4 + 2 * tvl) * 17 + p] + red[(kr * 4 + 2 * tvl + 1) * 17 + p];
    a.zpart[slot * 32 + pl] = static_cast<float>(z);
    if (pl == 0) {
      double g = 0.0;
      for (int k2 = 2 * tkl; k2 < 2 * tkl + 2; ++k2)
        for (int q2 = 2 * tvl; q2 < 2 * tvl + 2; ++q2) g += red[(k2 * 4 + q2) * 17 + 16];
      a.gpart[slot] = g;
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, T_COLS);
  }
}

// The walks' operands as hi + lo bf16 pairs, rows padded to whole chunks:
//   qb[bh][t] = γ^{j+1} R(t) q_t,   kf[bh][t] = d_k^{-1/2} γ^{b_c−1−j} R(t) k_t   (t < L)
//   zero for L ≤ t < Lp.  Thread ↔ (row of [BH·Lp], 8 columns).
template <typename Tin>
__global__ void __launch_bounds__(256) walk_prep_tc_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, __nv_bfloat16* __restrict__ qh,
    __nv_bfloat16* __restrict__ ql, __nv_bfloat16* __restrict__ kh, __nv_bfloat16* __restrict__ kl,
    const float2* __restrict__ cs, CallConsts cc, int H, int L, int Lp, int d_k, size_t rows) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int groups = d_k / 8;
  if (idx >= rows * groups) return;
  const size_t row = idx / groups;
  const int g = static_cast<int>(idx % groups);
  const int t = static_cast<int>(row % Lp);
  const size_t bh = row / Lp;
  const size_t o = row * d_k + 8 * g;
  if (t >= L) {
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(qh + o) = zero;
    *reinterpret_cast<uint4*>(ql + o) = zero;
    *reinterpret_cast<uint4*>(kh + o) = zero;
    *reinterpret_cast<uint4*>(kl + o) = zero;
    return;
  }
  const int h = static_cast<int>(bh % H);
  const int c = t / CH, j = t % CH;
  const int bc = min(CH, L - c * CH);
  const float wk = cc.kscale * exp2f(static_cast<float>(bc - 1 - j) * cc.lg2g[h]);
  const float wq = exp2f(static_cast<float>(j + 1) * cc.lg2g[h]);
  const size_t src = (bh * L + t) * static_cast<size_t>(d_k) + 8 * g;
  float xq[8], xk[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    xq[u] = to_f32(q[src + u]);
    xk[u] = to_f32(k[src + u]);
  }
  float oq[8], ok[8];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 e = cs[static_cast<size_t>(t) * (d_k / 2) + 4 * g + u];
    oq[2 * u] = wq * fmaf(xq[2 * u], e.x, -xq[2 * u + 1] * e.y);
    oq[2 * u + 1] = wq * fmaf(xq[2 * u + 1], e.x, xq[2 * u] * e.y);
    ok[2 * u] = wk * fmaf(xk[2 * u], e.x, -xk[2 * u + 1] * e.y);
    ok[2 * u + 1] = wk * fmaf(xk[2 * u + 1], e.x, xk[2 * u] * e.y);
  }
  // x = hi + lo: hi = bf16(x), lo = bf16(x − hi)
  auto split = [](const float (&x)[8], uint4& hi, uint4& lo) {
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ph[u] = pack_bf16x2(x[2 * u], x[2 * u + 1]);
      pl[u] = pack_bf16x2(x[2 * u] - bf16lo_to_f32(ph[u]), x[2 * u + 1] - bf16hi_to_f32(ph[u]));
    }
    hi = make_uint4(ph[0], ph[1], ph[2], ph[3]);
    lo = make_uint4(pl[0], pl[1], pl[2], pl[3]);
  };
  uint4 hq, lq, hk, lk;
  split(oq, hq, lq);
  split(ok, hk, lk);
  *reinterpret_cast<uint4*>(qh + o) = hq;
  *reinterpret_cast<uint4*>(ql + o) = lq;
  *reinterpret_cast<uint4*>(kh + o) = hk;
  *reinterpret_cast<uint4*>(kl + o) = lk;
}

}  // namespace tcw
}  // namespace ret
