// Parallel form of retention on the tensor cores (tcgen05, TMEM, TMA).
//
// Form («从RoPE到Retention…» §4.1; RetNet 保留网络 explainer 并行表征):
//   O = (Q′K′ᵀ ⊙ D) V + γ^{n+1} q′_n S_in,   D_nm = γ^{n−m} (n ≥ m), 0 otherwise.
// Tiled over 128-row blocks: query block i (rows n = 128i + r) against key
// blocks j ≤ i (columns m = 128j + c).  With the front pass's K̂′_m =
// ζ_c k′_m (ζ_c = γ^{127−c}) and ω_r = γ^{r+1−128} applied at the store,
//   D_nm = γ^{128(i−j)} · ω_r · ζ_c,
// so block (i, j) contributes ω ⊙ (g_ij · Q′_i K̂′_jᵀ) V_j with the scalar
// g_ij = γ^{128(i−j)}, and the diagonal block also takes the causal compare
// (c ≤ r, exact zeros above).  The state_in term is ω_r (Q′_i Ŝ_i)_r with
// Ŝ_i = bf16(γ^{128(i+1)} S_in).  The mask is never formed in memory.
//
// One CTA per (128-wide d_v tile, b·h, query block i); it walks j = 0 … i.
// Transposed products keep d_v on the TMEM lanes (as in the chunkwise
// kernel):  P̂ [r × c] = Q′_i K̂′_jᵀ into X;  Õᵀ [v × r] (+)= Ŝᵀ Q′_iᵀ and
// += V_jᵀ P̂ᵀ into O.  TMEM: X = [0,128), O = [128,256), SH = [256, 256+d_k/2).
#pragma once

#include "common.cuh"
#include "tc_primitives.cuh"

namespace ret {
namespace tcp {

using namespace ret::tc;

constexpr int CH = 128;               // block rows / columns
constexpr int VT = 128;               // d_v columns per CTA
constexpr int NCW = 16;               // drain warps
constexpr int NTHREADS = (NCW + 2) * 32;

enum Bar : int {
  Q_FULL = 0, K_FULL, V_FULL,         // TMA → MMA
  K_EMPTY, V_EMPTY,                   // MMA → TMA
  P_FULL,                             // QK of block j done   (MMA → drain)
  X_FREE,                             // P read out of X       (drain → MMA)
  P_SMEM,                             // P̂ in shared memory    (drain → MMA)
  PS_FREE,                            // PV done, P̂ reusable   (MMA → drain)
  SH_READY,                           // Ŝ_i written          (drain → MMA)
  O_FULL,                             // all products done     (MMA → drain)
  MMA_DONE, NBAR_
};

template <int DK>
struct Cfg {
  static_assert(DK == 64 || DK == 128 || DK == 256, "d_k");
  static constexpr int QBOX = DK / 64;
  static constexpr int SPT = DK / 4;              // state values per drain thread
  static constexpr uint32_t BOX = CH * 64 * 2;    // 16 KB
  static constexpr uint32_t Q_BYTES = CH * DK * 2;
  static constexpr uint32_t V_BYTES = CH * VT * 2;
  static constexpr uint32_t P_BYTES = CH * CH * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + Q_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + V_BYTES;
  static constexpr uint32_t OFF_OMEGA = OFF_P + P_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_OMEGA + CH * 4;
  static constexpr uint32_t OFF_TPTR = OFF_BAR + NBAR_ * 8;
  static constexpr uint32_t USED = OFF_TPTR + 16;
  static constexpr uint32_t SMEM_BYTES = USED + 1024;
  static constexpr uint32_t T_X = 0, T_O = 128, T_SH = 256;
  static constexpr uint32_t T_COLS = (256 + DK / 2) <= 256 ? 256 : 512;
};

struct ParArgs {
  const float* state_in;   // [BH][DK][d_v] or nullptr
  void* out;               // [BH][L][d_v] bf16, or fp32 when out_f32
  int out_f32;
  int H, L, d_v;
};

// grid = (d_v / 128, B·H, L / 128); block = 576 threads; 1 CTA per SM.
template <int DK>
__global__ void __launch_bounds__(NTHREADS, 1)
    parallel_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, ParArgs args, CallConsts cc) {
  using C = Cfg<DK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V, sP = sb + C::OFF_P;
  float* omega = reinterpret_cast<float*>(smem + C::OFF_OMEGA);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v0 = blockIdx.x * VT;
  const int bh = blockIdx.y;
  const int qb = blockIdx.z;                 // query block i
  const int h = bh % args.H;
  const int L = args.L, d_v = args.d_v;
  const int nkb = qb + 1;                    // key blocks j = 0 … i
  const bool has_state = args.state_in != nullptr;
  const float lg2 = cc.lg2g[h];

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int i = 0; i < NBAR_; ++i) {
      const bool from_drain = (i == X_FREE || i == P_SMEM || i == SH_READY);
      mbar_init(bar(i), from_drain ? NCW : 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + C::OFF_TPTR, C::T_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x < CH) omega[threadIdx.x] = gpow(lg2, static_cast<float>(static_cast<int>(threadIdx.x) + 1 - CH));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_TPTR);

  if (warp == 0) {
    // ------------------------------ TMA producer ---------------------------
    if (lane == 0) {
      const int yq = bh * L + qb * CH;
      mbar_arrive_expect_tx(bar(Q_FULL), C::Q_BYTES);
      for (int b = 0; b < C::QBOX; ++b) tma_load_2d(sQ + b * C::BOX, &tm_q, 64 * b, yq, bar(Q_FULL));
      int issued = -1;
      for (int j = 0; j < nkb; ++j) {
        const uint32_t pp = static_cast<uint32_t>(j - 1) & 1u;
        const int y = bh * L + j * CH;
        if (j > 0 && !mbar_wait(bar(K_EMPTY), pp, 0x501)) break;
        mbar_arrive_expect_tx(bar(K_FULL), C::Q_BYTES);
        for (int b = 0; b < C::QBOX; ++b) tma_load_2d(sK + b * C::BOX, &tm_k, 64 * b, y, bar(K_FULL));
        if (j > 0 && !mbar_wait(bar(V_EMPTY), pp, 0x502)) break;
        mbar_arrive_expect_tx(bar(V_FULL), C::V_BYTES);
        for (int b = 0; b < 2; ++b) tma_load_2d(sV + b * C::BOX, &tm_v, v0 + 64 * b, y, bar(V_FULL));
        issued = j;
      }
      if (status_aborted()) {   // never leave bulk copies landing after exit
        mbar_wait(bar(Q_FULL), 0, 0x5f0, kWaitBudgetCycles / 8);
        if (issued >= 0) {
          const uint32_t pl = static_cast<uint32_t>(issued) & 1u;
          mbar_wait(bar(K_FULL), pl, 0x5f1, kWaitBudgetCycles / 8);
          mbar_wait(bar(V_FULL), pl, 0x5f2, kWaitBudgetCycles / 8);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer -----------------------------
    if (lane == 0) {
      const uint32_t tX = tmem + C::T_X, tO = tmem + C::T_O, tSH = tmem + C::T_SH;
      constexpr uint32_t ID_P = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t ID_QS = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t ID_PV = idesc_bf16_f32(128, 128, 1, 0);
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK = sdesc_sw128(sK, 16, 1024);
      const uint64_t dV = sdesc_sw128(sV, C::BOX, 1024);
      const uint64_t dP = sdesc_sw128(sP, 16, 1024);
      auto kmaj = [](int s) -> uint64_t {
        return static_cast<uint64_t>(((s >> 2) * C::BOX + (s & 3) * 32) >> 4);
      };
      bool ok = mbar_wait(bar(Q_FULL), 0, 0x601);
      if (ok && has_state) {   // Õᵀ = Ŝ_iᵀ Q′_iᵀ
        ok = mbar_wait(bar(SH_READY), 0, 0x602);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int s = 0; s < DK / 16; ++s) mma_ts(tO, tSH + s * 8, dQ + kmaj(s), ID_QS, s > 0 ? 1u : 0u);
        }
      }
      for (int j = 0; ok && j < nkb; ++j) {
        const uint32_t pj = static_cast<uint32_t>(j) & 1u;
        const uint32_t pp = static_cast<uint32_t>(j - 1) & 1u;
        // P = Q′_i K̂′_jᵀ into X (needs the previous P read out)
        if (!mbar_wait(bar(K_FULL), pj, 0x603)) break;
        if (j > 0 && !mbar_wait(bar(X_FREE), pp, 0x604)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < DK / 16; ++s) mma_ss(tX, dQ + kmaj(s), dK + kmaj(s), ID_P, s > 0 ? 1u : 0u);
        mma_commit(bar(P_FULL));
        mma_commit(bar(K_EMPTY));
        // Õᵀ += V_jᵀ P̂ᵀ (needs the scaled, masked bf16 P̂ in shared memory)
        if (!mbar_wait(bar(V_FULL), pj, 0x605)) break;
        if (!mbar_wait(bar(P_SMEM), pj, 0x606)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < CH / 16; ++s)
          mma_ss(tO, dV + static_cast<uint64_t>(s * 128), dP + kmaj(s), ID_PV,
                 (has_state || j > 0 || s > 0) ? 1u : 0u);
        mma_commit(bar(PS_FREE));
        mma_commit(bar(V_EMPTY));
      }
      mma_commit(bar(O_FULL));
      mma_commit(bar(MMA_DONE));
      mbar_wait(bar(MMA_DONE), 0, 0x6ff);
    }
  } else {
    // ------------------------------ drain warps ----------------------------
    const int w = warp - 2;                 // 0..15
    const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
    const int cs = w >> 2;                  // 32-column slice
    const int kr = w >> 2;                  // state k range [kr*SPT, kr*SPT+SPT)
    const int vl = 32 * quarter + lane;     // TMEM lane: v for Õ / Ŝ, r for P
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    bool ok = true;

    if (has_state) {   // Ŝ_i = bf16(γ^{128(i+1)} S_in) for this thread's v lane and k range
      const float gs = gpow(lg2, static_cast<float>(CH * (qb + 1)));
      const float* sin = args.state_in + static_cast<size_t>(bh) * DK * d_v + v0 + vl;
#pragma unroll
      for (int c = 0; c < C::SPT / 16; ++c) {
        uint32_t pk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int kk = kr * C::SPT + c * 16 + 2 * u;
          pk[u] = pack_bf16x2(gs * sin[static_cast<size_t>(kk) * d_v], gs * sin[static_cast<size_t>(kk + 1) * d_v]);
        }
        tmem_st8(tmem + C::T_SH + lane_off + (kr * C::SPT + c * 16) / 2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SH_READY));
    }

    for (int j = 0; j < nkb && ok; ++j) {
      const uint32_t pj = static_cast<uint32_t>(j) & 1u;
      const uint32_t pp = static_cast<uint32_t>(j - 1) & 1u;
      if (!mbar_wait(bar(P_FULL), pj, 0x701)) { ok = false; break; }
      tc_fence_after();
      const float g = gpow(lg2, static_cast<float>(CH * (qb - j)));   // γ^{128(i−j)}
      const bool diag = (j == qb);
      const int r = vl;   // row of P = TMEM lane
      uint32_t pk[2][8];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t x[16];
        tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&x[0]));
        tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 16 * hf + 8, *reinterpret_cast<uint32_t(*)[8]>(&x[8]));
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = 32 * cs + 16 * hf + 2 * u;
          const float a = (!diag || c <= r) ? g * __uint_as_float(x[2 * u]) : 0.f;
          const float b = (!diag || c + 1 <= r) ? g * __uint_as_float(x[2 * u + 1]) : 0.f;
          pk[hf][u] = pack_bf16x2(a, b);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(X_FREE));
      // P̂ of block j − 1 must have been consumed by its PV before overwriting
      if (j > 0 && !mbar_wait(bar(PS_FREE), pp, 0x702)) { ok = false; break; }
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        const int c0 = 32 * cs + 8 * g8;
        const uint32_t* pw = &pk[g8 >> 1][(g8 & 1) * 4];
        st_shared_v4(sP + (c0 >> 6) * C::BOX + sw128_offset(r, c0 & 63), pw[0], pw[1], pw[2], pw[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P_SMEM));
    }

    if (ok && mbar_wait(bar(O_FULL), 0, 0x703)) {
      tc_fence_after();
      const size_t base = (static_cast<size_t>(bh) * L + static_cast<size_t>(qb) * CH + 32 * cs) * d_v + v0 + vl;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t x[16];
        tmem_ld8(tmem + C::T_O + lane_off + 32 * cs + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&x[0]));
        tmem_ld8(tmem + C::T_O + lane_off + 32 * cs + 16 * hf + 8, *reinterpret_cast<uint32_t(*)[8]>(&x[8]));
        tmem_ld_wait();
        const size_t gb0 = base + static_cast<size_t>(16 * hf) * d_v;
        if (args.out_f32) {
          float* o = reinterpret_cast<float*>(args.out) + gb0;
#pragma unroll
          for (int c = 0; c < 16; ++c)
            o[static_cast<size_t>(c) * d_v] = omega[32 * cs + 16 * hf + c] * __uint_as_float(x[c]);
        } else {
          __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(args.out) + gb0;
#pragma unroll
          for (int c = 0; c < 16; ++c)
            o[static_cast<size_t>(c) * d_v] =
                __float2bfloat16_rn(omega[32 * cs + 16 * hf + c] * __uint_as_float(x[c]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::T_COLS);
  }
}

}  // namespace tcp
}  // namespace ret
