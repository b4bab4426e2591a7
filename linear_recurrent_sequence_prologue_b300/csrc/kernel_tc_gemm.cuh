// Projection GEMMs of the MSR block on tcgen05 CTA pairs.
//
// The block around the retention core (the SimpleRetention of «RetNet：
// Transformer的革命性继任者？»: q = X·W_Q, k = X·W_K, v = X·W_V per head; the
// gate and output projection of the published MSR block, reading 15 of the
// design notes) is five dense contractions C[M×N] = A[M×K]·W[K×N] with
// A = X or the gated, normalised retention output (row-major, K contiguous)
// and W row-major (N contiguous).  One kernel runs them all:
//
//   * a cluster of two CTAs owns a 256 × 256 tile of C; each CTA stages its
//     128 rows of A (K-major, 128-byte swizzle) and its 128 columns of W
//     (MN-major) per 64-wide K step, three steps in flight, and the even CTA
//     issues one pair MMA (tcgen05.mma.cta_group::2, M = 256, N = 256) per
//     16 of K into both CTAs' tensor memory (each CTA gets its 128 rows × 256
//     columns of the fp32 accumulator);
//   * four epilogue warps per CTA read the accumulator (one row per thread,
//     32 columns per tcgen05.ld) and store it through one of the modes below;
//   * two CTAs fit on one SM (96 KB of shared memory and 256 TMEM columns
//     each), so one tile's epilogue overlaps another tile's MMAs.
//
// Epilogue modes (columns n = h·dh + c of head h, rows m = b·L + t):
//   PLAIN  C as it is, bf16 or fp32 [M][N];
//   HEADS  bf16 into the head layout [(b·H + h)·L + t][c] (v);
//   ROT_Q  Q″ for the chunk kernels: the bf16 product rotated by R((pos0+t)θ)
//          and multiplied by ω_{t mod 128}, into [(b·H + h)·Lp + t][c];
//   ROT_K  K̂′: rotated, times d_k^{-1/2}·ζ_{t mod 128}, same layout.
// The ROT modes round the product to bf16 first and then apply the front
// pass's own arithmetic (rot_q_word / rot_k_word / row_factors, angles from a
// table filled by angle_cs), so Q″ and K̂′ are the bits that the front pass
// would write from a bf16 q, k = X·W.
#pragma once

#include "common.cuh"
#include "tc_primitives.cuh"
#include "kernel_tc_chunk.cuh"

namespace ret {
namespace tcg {

using namespace ret::tc;
using tcc::rot_k_word;
using tcc::rot_q_word;
using tcc::row_factors;

constexpr int BM = 128;                              // rows of C per CTA (256 per pair)
constexpr int BN = 256;                              // columns of C per pair
constexpr int BK = 64;                               // K per stage
constexpr int STAGES = 3;
constexpr int NEPI = 4;                              // epilogue warps
constexpr int NTHREADS = (2 + NEPI) * 32;
constexpr uint32_t A_BYTES = BM * BK * 2;            // 16 KB: 128 rows × 64 K
constexpr uint32_t BBOX = BK * 64 * 2;               // 8 KB: 64 K rows × 64 columns
constexpr uint32_t B_BYTES = 2 * BBOX;               // this CTA's 128 columns
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB
enum Bar : int { FULL0 = 0, EMPTY0 = STAGES, ACC_FULL = 2 * STAGES, NBAR_ };
constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
constexpr uint32_t OFF_TPTR = OFF_BAR + NBAR_ * 8;
constexpr uint32_t SMEM_BYTES = OFF_TPTR + 16 + 1024;   // + slack for 1024-B alignment
constexpr uint32_t T_COLS = 256;

enum Mode : int { PLAIN = 0, HEADS = 1, ROT_Q = 2, ROT_K = 3 };

struct GemmArgs {
  int M = 0, N = 0, K = 0;
  void* out = nullptr;          // see the modes
  int out_f32 = 0;              // PLAIN only
  int L = 0, Lp = 0, H = 0, dh = 0;   // HEADS / ROT_*: tokens per sequence, rows per head, heads, width
  float pos0 = 0.f;             // ROT_*: position of token 0
  const float2* cs = nullptr;   // ROT_*: (cos, sin) of (pos0 + t)·θ_i, [L][dh/2]
};

// grid = (2·⌈M/256⌉, N/256), cluster = (2, 1, 1), block = 192 threads.
// Warp 0: TMA (both CTAs).  Warp 1: TMEM allocation; its lane 0 of the even
// CTA issues the pair MMAs.  Warps 2..5: epilogue.
template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 2)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,   // A [M][K], boxes 64 × 128
                     const __grid_constant__ CUtensorMap tm_w,   // W [K][N], boxes 64 × 64
                     GemmArgs g, CallConsts cc) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto sA = [&](int s) { return sb + static_cast<uint32_t>(s) * STAGE_BYTES; };
  auto sB = [&](int s) { return sb + static_cast<uint32_t>(s) * STAGE_BYTES + A_BYTES; };
  auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const uint32_t lead_bar0 = mapa_shared(bar(0), 0);
  auto lead_bar = [&](int i) -> uint32_t { return lead_bar0 + 8u * static_cast<uint32_t>(i); };

  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = static_cast<int>(blockIdx.x >> 1) * 2 * BM + BM * static_cast<int>(rank);   // this CTA's rows
  const int n0 = static_cast<int>(blockIdx.y) * BN;                                          // the pair's columns
  const int nk = g.K / BK;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_w);
    for (int i = 0; i < NBAR_; ++i) mbar_init(bar(i), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(sb + OFF_TPTR, T_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TPTR);

  if (warp == 0) {
    // ------------------------------ TMA ----------------------------------
    if (lane == 0) {
      int issued = -1;
      for (int k = 0; k < nk; ++k) {
        const int s = k % STAGES;
        if (k >= STAGES && !mbar_wait(bar(EMPTY0 + s), static_cast<uint32_t>(k / STAGES - 1) & 1u, 0x601))
          break;
        if (rank == 0) mbar_arrive_expect_tx(bar(FULL0 + s), 2 * STAGE_BYTES);
        tma_load_2d_pair(sA(s), &tm_a, k * BK, m0, lead_bar(FULL0 + s));
        for (int b = 0; b < 2; ++b)
          tma_load_2d_pair(sB(s) + b * BBOX, &tm_w, n0 + 128 * static_cast<int>(rank) + 64 * b, k * BK,
                           lead_bar(FULL0 + s));
        issued = k;
      }
      // Never leave with copies still landing (the even CTA counts both CTAs' bytes).
      if (rank == 0 && issued >= 0 && status_aborted())
        for (int k = issued - STAGES + 1 > 0 ? issued - STAGES + 1 : 0; k <= issued; ++k)
          mbar_wait(bar(FULL0 + k % STAGES), static_cast<uint32_t>(k / STAGES) & 1u, 0x6f0,
                    kWaitBudgetCycles / 16);
    }
  } else if (warp == 1) {
    // ------------------------------ MMA ----------------------------------
    if (lane == 0 && rank == 0) {
      constexpr uint32_t ID = idesc_bf16_f32(256, 256, 0, 1);   // A K-major, W MN-major
      bool ok = true;
      for (int k = 0; k < nk && ok; ++k) {
        const int s = k % STAGES;
        if (!mbar_wait_cl(bar(FULL0 + s), static_cast<uint32_t>(k / STAGES) & 1u, 0x602)) { ok = false; break; }
        tc_fence_after();
        const uint64_t da = sdesc_sw128(sA(s), 16, 1024);      // 128-B rows of 64 K
        const uint64_t dw = sdesc_sw128(sB(s), BBOX, 1024);    // 64-column groups BBOX apart
#pragma unroll
        for (int j = 0; j < BK / 16; ++j)   // A: +32 B per 16 of K; W: +16 rows of 128 B
          mma_ss_pair(tmem, da + static_cast<uint64_t>(2 * j), dw + static_cast<uint64_t>(128 * j), ID,
                      (k > 0 || j > 0) ? 1u : 0u);
        mma_commit_pair(bar(EMPTY0 + s));
      }
      // The accumulator is complete once every issued MMA is (both CTAs' barriers).
      mma_commit_pair(bar(ACC_FULL));
    }
  } else {
    // ---------------------------- epilogue -------------------------------
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;   // TMEM lane = row of this CTA's 128
    const int m = m0 + row;
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    const bool ok = mbar_wait(bar(ACC_FULL), 0, 0x603);
    tc_fence_after();
    if (ok) {
      int b = 0, t = 0;
      if (MODE != PLAIN) { b = m / g.L; t = m - b * g.L; }
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        __syncwarp();   // tcgen05.ld is warp-collective: the whole warp, converged
        tmem_ld32(tmem + lane_off + 32 * c, r);
        tmem_ld_wait();
        if (m >= g.M) continue;   // rows past M: nothing to store (after the load)
        const int n = n0 + 32 * c;
        if constexpr (MODE == PLAIN) {
          if (g.out_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(g.out) + static_cast<size_t>(m) * g.N + n);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              o[u] = make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                 __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3]));
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.out) + static_cast<size_t>(m) * g.N + n);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              o[u] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * u]), __uint_as_float(r[8 * u + 1])),
                                pack_bf16x2(__uint_as_float(r[8 * u + 2]), __uint_as_float(r[8 * u + 3])),
                                pack_bf16x2(__uint_as_float(r[8 * u + 4]), __uint_as_float(r[8 * u + 5])),
                                pack_bf16x2(__uint_as_float(r[8 * u + 6]), __uint_as_float(r[8 * u + 7])));
          }
        } else {
          const int h = n / g.dh, cc0 = n - h * g.dh;
          const size_t rowi = static_cast<size_t>(b * g.H + h) * (MODE == HEADS ? g.L : g.Lp) + t;
          uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.out) + rowi * g.dh + cc0);
          uint32_t w[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) w[u] = pack_bf16x2(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
          if constexpr (MODE == ROT_Q || MODE == ROT_K) {
            float zk, wq;
            row_factors(cc, h, t, g.L, g.Lp, tcc::CH, 1, zk, wq);
            const float4* csr = reinterpret_cast<const float4*>(g.cs + static_cast<size_t>(t) * (g.dh / 2) + cc0 / 2);
#pragma unroll
            for (int u = 0; u < 8; ++u) {   // pairs 2u, 2u + 1 of this 32-column slice
              const float4 a = __ldg(csr + u);
              if constexpr (MODE == ROT_Q) {
                w[2 * u] = rot_q_word(w[2 * u], a.x, a.y, wq);
                w[2 * u + 1] = rot_q_word(w[2 * u + 1], a.z, a.w, wq);
              } else {
                w[2 * u] = rot_k_word(w[2 * u], __fmul_rn(zk, a.x), __fmul_rn(zk, a.y));
                w[2 * u + 1] = rot_k_word(w[2 * u + 1], __fmul_rn(zk, a.z), __fmul_rn(zk, a.w));
              }
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) o[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
    }
  }

  // Neither CTA leaves (or frees its TMEM) while the pair's MMAs or copies
  // may still touch it.
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, T_COLS);
  }
}

// ---------------------------------------------------------------------------
// GroupNorm of the retention output and the swish gate, per token and head:
//   a[b·L + t][h·d_v + v] = swish(g[b·L + t][h·d_v + v]) · GN(o[(b·H + h)·L + t])[v]
// with GN over the head's d_v channels (biased variance, eps) and
// swish(x) = x·σ(x).  o fp32 [B·H·L][d_v]; g, a bf16 [B·L][H·d_v].  One warp
// per (b, h, t); d_v a multiple of 8.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gn_gate_kernel(const float* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ gate,
                                                      __nv_bfloat16* __restrict__ a, int H, int L,
                                                      int d_v, size_t rows, float eps) {
  const size_t row = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const size_t bh = row / L;
  const int t = static_cast<int>(row - bh * L);
  const int h = static_cast<int>(bh % H);
  const size_t b = bh / H;
  const float* xr = o + row * d_v;
  float s = 0.f;
  for (int c = 4 * lane; c < d_v; c += 128) {
    const float4 x4 = *reinterpret_cast<const float4*>(xr + c);
    s += (x4.x + x4.y) + (x4.z + x4.w);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  const float mu = s / static_cast<float>(d_v);
  float q = 0.f;
  for (int c = 4 * lane; c < d_v; c += 128) {
    const float4 x4 = *reinterpret_cast<const float4*>(xr + c);
    q = fmaf(x4.x - mu, x4.x - mu, q);
    q = fmaf(x4.y - mu, x4.y - mu, q);
    q = fmaf(x4.z - mu, x4.z - mu, q);
    q = fmaf(x4.w - mu, x4.w - mu, q);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) q += __shfl_xor_sync(0xffffffffu, q, off);
  const float rstd = rsqrtf(q / static_cast<float>(d_v) + eps);
  const size_t arow = (b * L + t) * static_cast<size_t>(H) * d_v + static_cast<size_t>(h) * d_v;
  for (int c = 4 * lane; c < d_v; c += 128) {
    const float4 x4 = *reinterpret_cast<const float4*>(xr + c);
    const uint2 g2 = *reinterpret_cast<const uint2*>(gate + arow + c);
    const float gx[4] = {bf16lo_to_f32(g2.x), bf16hi_to_f32(g2.x), bf16lo_to_f32(g2.y), bf16hi_to_f32(g2.y)};
    const float xv[4] = {x4.x, x4.y, x4.z, x4.w};
    float y[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float sw = gx[u] / (1.f + __expf(-gx[u]));   // swish(x) = x·σ(x)
      y[u] = sw * ((xv[u] - mu) * rstd);
    }
    *reinterpret_cast<uint2*>(a + arow + c) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
  }
}

}  // namespace tcg
}  // namespace ret
