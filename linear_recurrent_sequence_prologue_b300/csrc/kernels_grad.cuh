// Parameter gradients of the retention core (γ per head, θ per rotation
// pair), and the GroupNorm forward (row-staged) and backward.
//
// dγ_h, dθ_i.  Both are sums over (query n, key m) pairs of the decay- or
// angle-weighted terms of <dO, out> + <dS_out, S_out> («从RoPE到Retention…»
// §2-§4: ∂γ^{n−m}/∂γ = (n−m)·γ^{n−m−1}; θ is learnable, and pair i of
// q′_t, k′_t is rotated by (pos0 + t)·θ_i, so the angle of a pair's score
// moves with (m − n)).  Written with positions over the whole sequence
// (Σ_t t·(dO_t·o_t − v_t·dv_t) for γ) the weights grow with L while the
// result only grows with the decay window, and the two big sums cancel: the
// rounding of bf16 operands would be amplified by L / window.  So the sums
// are split at chunk boundaries (chunks of b = 128 tokens, c = 0..C−1, the
// last of r tokens; S_c the state after chunk c, dS_c its gradient, S_{−1} =
// S_in, dS_{C−1} = dS_out; j the index inside a chunk, κ = (b−1)/2).  Reverse
// mode through the chunk recurrence (o_j = Σ_{i≤j} γ^{j−i}(q′_j·k′_i)v_i +
// γ^{j+1}q′_j S_{c−1}, S_c = γ^{b_c}S_{c−1} + Σ_i γ^{b_c−1−i}k′_iᵀv_i) gives
//   γ·dγ = Σ_t (j−κ)·(dO_t·o_t − v_t·dv_t) + (1+κ)<S_{−1}, dS_{−1}>
//          + (r−1−κ)<S_{C−1}, dS_{C−1}> + b·Σ_{c=0}^{C−2} <S_c, dS_c>
//   dθ_i = Σ_t (j−κ)·(dq_t·J q_t + dk_t·J k_t)_i + (pos0+κ)·Z_{−1,i}
//          − (pos0+(C−1)b+κ)·Z_{C−1,i} + b·Σ_{c=0}^{C−2} Z_{c,i}
// with J(a, b) = (−b, a) on each pair (dQ′·J q′ = dq·J q since J commutes
// with the rotation) and Z_{c,i} = Σ_v (S_c[2i+1,v]·dS_c[2i,v] −
// S_c[2i,v]·dS_c[2i+1,v]).  Every weight is now at most b or is the genuine
// absolute-position weight of the state terms.  The row sums use the
// caller's out, dv, dq, dk; the states are recomputed here in fp32 from q,
// k, v, d_out (a forward walk stores S_c, a backward walk carries dS_c and
// forms the boundary products), so they carry no bf16 rounding.
//
// GroupNorm backward (one group per (b, h, t) row over d_v channels, biased
// variance, «从RoPE到Retention…» §5): with x̂ = (x − μ)·rstd and g = dy ⊙ w,
//   dx = rstd·(g − mean(g) − x̂·mean(g ⊙ x̂)),  dw = Σ_rows dy ⊙ x̂,  db = Σ_rows dy.
//
// Every reduction writes per-block partials that a finishing kernel sums in
// a fixed order (in double), so the results do not depend on scheduling.
#pragma once

#include "common.cuh"

namespace ret {
namespace grad {

constexpr int kRowsPerBlock = 64;
constexpr int kGradChunk = 128;                         // b of the boundary split
constexpr float kKappa = 0.5f * (kGradChunk - 1);      // κ, exact in fp32

// 8 consecutive row elements as fp32: one 16-byte load for bf16, two for fp32.
template <typename T> __device__ __forceinline__ void load8(const T* p, float (&x)[8]);
template <> __device__ __forceinline__ void load8<float>(const float* p, float (&x)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <> __device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16lo_to_f32(w[i]);
    x[2 * i + 1] = bf16hi_to_f32(w[i]);
  }
}

template <typename T> __device__ __forceinline__ void store8(T* p, const float (&x)[8]);
template <> __device__ __forceinline__ void store8<float>(float* p, const float (&x)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}
template <> __device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float (&x)[8]) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                            pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
}

// Per-thread asynchronous 16-byte copies global → shared (waited for with
// cp.async.wait_group by the copying thread).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <typename Tx>
__device__ __forceinline__ void lds8(const Tx* p, float (&x)[8]);
template <> __device__ __forceinline__ void lds8<float>(const float* p, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <> __device__ __forceinline__ void lds8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) { x[2 * i] = bf16lo_to_f32(w[i]); x[2 * i + 1] = bf16hi_to_f32(w[i]); }
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// ---------------------------------------------------------------------------
// Row pass of the parameter gradients.  Block = (b, h, segment of
// kRowsPerBlock tokens), 8 warps, warp w takes tokens w, w + 8, …  Writes
// gpart[block] (the segment's Σ (j−κ)·(dO·o − v·dv), double) and
// tpart[i][block] (the segment's Σ (j−κ)·(dq·J q + dk·J k)_i; pair-major, so
// the finishing sums read it contiguously), j = t mod kGradChunk.  VEC: d_k and d_v are multiples of 8 (rows
// read as 16-byte vectors); otherwise element by element.
// ---------------------------------------------------------------------------
struct ParamArgs {
  const void* q; const void* k; const void* v; const void* d_out;
  const void* out; const void* dq; const void* dk; const void* dv;
  int H, L, d_k, d_v, nseg;
  double* gpart;       // [B·H·nseg] or null (no dγ)
  float* tpart;        // [d_k/2][B·H·nseg] or null (no dθ)
};

template <typename Tin, typename Tout, typename Tg, bool VEC>
__global__ void __launch_bounds__(256) param_rows_kernel(ParamArgs a) {
  __shared__ float tred[8][kMaxPairs];
  __shared__ double gred[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x % a.nseg;
  const size_t bh = blockIdx.x / a.nseg;
  const int P = a.d_k / 2;
  const int t0 = seg * kRowsPerBlock, t1 = min(a.L, t0 + kRowsPerBlock);
  float gacc = 0.f;
  float tacc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) tacc[j] = 0.f;

  for (int t = t0 + warp; t < t1; t += 8) {
    const size_t row = bh * a.L + t;
    if (a.gpart) {   // this lane's share of dO_t·o_t − v_t·dv_t
      const Tin* dO = static_cast<const Tin*>(a.d_out) + row * a.d_v;
      const Tout* o = static_cast<const Tout*>(a.out) + row * a.d_v;
      const Tin* v = static_cast<const Tin*>(a.v) + row * a.d_v;
      const Tg* dv = static_cast<const Tg*>(a.dv) + row * a.d_v;
      float s = 0.f;
      if (VEC) {
        for (int c = 8 * lane; c < a.d_v; c += 256) {
          float x0[8], x1[8], x2[8], x3[8];
          load8(dO + c, x0); load8(o + c, x1); load8(v + c, x2); load8(dv + c, x3);
#pragma unroll
          for (int e = 0; e < 8; ++e) s = fmaf(x0[e], x1[e], fmaf(-x2[e], x3[e], s));
        }
      } else {
        for (int c = lane; c < a.d_v; c += 32)
          s = fmaf(to_f32(dO[c]), to_f32(o[c]), fmaf(-to_f32(v[c]), to_f32(dv[c]), s));
      }
      gacc = fmaf(static_cast<float>(t % kGradChunk) - kKappa, s, gacc);
    }
    if (a.tpart) {
      const float pos = static_cast<float>(t % kGradChunk) - kKappa;
      const Tin* q = static_cast<const Tin*>(a.q) + row * a.d_k;
      const Tin* k = static_cast<const Tin*>(a.k) + row * a.d_k;
      const Tg* dq = static_cast<const Tg*>(a.dq) + row * a.d_k;
      const Tg* dk = static_cast<const Tg*>(a.dk) + row * a.d_k;
      if (VEC) {   // lane owns pairs 4·(lane + 32j) … +3, j = 0, 1
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = 8 * (lane + 32 * j);
          if (c < a.d_k) {
            float xq[8], xk[8], gq[8], gk[8];
            load8(q + c, xq); load8(k + c, xk); load8(dq + c, gq); load8(dk + c, gk);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const float term = fmaf(gq[2 * p + 1], xq[2 * p], -gq[2 * p] * xq[2 * p + 1]) +
                                 fmaf(gk[2 * p + 1], xk[2 * p], -gk[2 * p] * xk[2 * p + 1]);
              tacc[4 * j + p] = fmaf(pos, term, tacc[4 * j + p]);
            }
          }
        }
      } else {     // lane owns pairs lane + 32j, j < 8
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = lane + 32 * j;
          if (i < P) {
            const float q0 = to_f32(q[2 * i]), q1 = to_f32(q[2 * i + 1]);
            const float k0 = to_f32(k[2 * i]), k1 = to_f32(k[2 * i + 1]);
            const float term = fmaf(to_f32(dq[2 * i + 1]), q0, -to_f32(dq[2 * i]) * q1) +
                               fmaf(to_f32(dk[2 * i + 1]), k0, -to_f32(dk[2 * i]) * k1);
            tacc[j] = fmaf(pos, term, tacc[j]);
          }
        }
      }
    }
  }

  if (a.gpart) {
    const float w = warp_sum(gacc);
    if (lane == 0) gred[warp] = static_cast<double>(w);
  }
  if (a.tpart) {
    if (VEC) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int i = 4 * (lane + 32 * j) + p;
          if (i < P) tred[warp][i] = tacc[4 * j + p];
        }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (lane + 32 * j < P) tred[warp][lane + 32 * j] = tacc[j];
    }
  }
  __syncthreads();
  if (a.gpart && threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < 8; ++w) s += gred[w];
    a.gpart[blockIdx.x] = s;
  }
  if (a.tpart)
    for (int i = threadIdx.x; i < P; i += 256) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) s += tred[w][i];
      a.tpart[static_cast<size_t>(i) * gridDim.x + blockIdx.x] = s;
    }
}

// ---------------------------------------------------------------------------
// State walks.  Block = (b, h, 64 × 64 tile of the d_k × d_v state), 256
// threads; thread (ty, tx) = (tid / 16, tid % 16) owns rows 4ty … 4ty+3 and
// columns 4tx … 4tx+3 of the tile (rows 4ty, 4ty+1 and 4ty+2, 4ty+3 are two
// rotation pairs).  A chunk's rank-b_c update Σ_i w_i a_iᵀ b_i is staged 32
// rows at a time in shared memory (a: the rotated, weighted k′ or q′ columns
// of the tile; b: the v or dO columns).  The angle table cs[t][i] holds
// (cos, sin) of (pos0 + t)·θ_i.  States are stored per (b, h, chunk, tile)
// in thread order, 16 floats per thread.
// ---------------------------------------------------------------------------
constexpr int kTile = 64;
constexpr int kStage = 32;

struct WalkArgs {
  const void* a;        // k (forward walk) or q (backward walk) [BH][L][d_k]
  const void* b;        // v or d_out [BH][L][d_v]
  const float* s0;      // forward: S_in; backward: dS_out [BH][d_k][d_v], or null
  const float* s_in;    // backward: S_in (the state before chunk 0), or null
  float* states;        // [BH][C][tiles][4096]: S_c written (forward), read (backward)
  const float2* cs;     // [L][d_k/2]
  double* gpart;        // backward: [BH·tiles] weighted Σ <S_c, dS_c>
  float* zpart;         // backward: [BH·tiles][32] weighted Σ Z_c per pair of the tile
  int H, L, d_k, d_v, C, ntk, ntv;
  float ascale;         // forward: d_k^{-1/2}; backward: 1
  float pos0;
  CallConsts cc;
};

// Stage rows t0 … t0+kStage−1 of chunk c (local indices j0 …) into As, Bs.
// Forward: weight γ^{b_c−1−j}; backward: γ^{j+1}.
template <typename Tin, bool FWD>
__device__ __forceinline__ void stage_rows(const WalkArgs& w, size_t bh, int h, int c, int bc, int j0,
                                           int k0, int v0, float (*As)[kTile + 4],
                                           float (*Bs)[kTile + 4]) {
  const Tin* A = static_cast<const Tin*>(w.a);
  const Tin* Bm = static_cast<const Tin*>(w.b);
  const int tid = threadIdx.x;
  const float lg = w.cc.lg2g[h];
  // a: kStage rows × 32 pairs; thread → (row tid / 8, pairs 4·(tid % 8) … +3)
  {
    const int r = tid >> 3, jl = j0 + r;
    const int t = c * kGradChunk + jl;
    const bool live = jl < bc;
    const float wgt = live ? w.ascale * exp2f((FWD ? static_cast<float>(bc - 1 - jl)
                                                   : static_cast<float>(jl + 1)) * lg) : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int pl = 4 * (tid & 7) + u;        // pair within the tile
      const int col = k0 + 2 * pl;
      float x0 = 0.f, x1 = 0.f;
      if (live && col < w.d_k) {
        const size_t off = (bh * w.L + t) * static_cast<size_t>(w.d_k) + col;
        const float2 e = w.cs[static_cast<size_t>(t) * (w.d_k / 2) + col / 2];
        const float a0 = to_f32(A[off]), a1 = to_f32(A[off + 1]);
        x0 = wgt * fmaf(a0, e.x, -a1 * e.y);   // rotate by the angle: (a0 c − a1 s, a1 c + a0 s)
        x1 = wgt * fmaf(a1, e.x, a0 * e.y);
      }
      As[r][2 * pl] = x0;
      As[r][2 * pl + 1] = x1;
    }
  }
  // b: kStage rows × 64 columns; thread → (row tid / 8, columns 8·(tid % 8) … +7)
  {
    const int r = tid >> 3, jl = j0 + r;
    const int t = c * kGradChunk + jl;
    const bool live = jl < bc;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int col = v0 + 8 * (tid & 7) + u;
      Bs[r][8 * (tid & 7) + u] =
          live && col < w.d_v ? to_f32(Bm[(bh * w.L + t) * static_cast<size_t>(w.d_v) + col]) : 0.f;
    }
  }
}

// acc (4 × 4 of the tile) += Σ over the chunk's rows of As[i][rows]ᵀ Bs[i][cols].
template <typename Tin, bool FWD>
__device__ __forceinline__ void chunk_update(const WalkArgs& w, size_t bh, int h, int c, int k0, int v0,
                                             float (&acc)[4][4], float (*As)[kTile + 4],
                                             float (*Bs)[kTile + 4]) {
  const int bc = min(kGradChunk, w.L - c * kGradChunk);
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  for (int j0 = 0; j0 < bc; j0 += kStage) {
    __syncthreads();
    stage_rows<Tin, FWD>(w, bh, h, c, bc, j0, k0, v0, As, Bs);
    __syncthreads();
#pragma unroll 8
    for (int i = 0; i < kStage; ++i) {
      const float4 a = *reinterpret_cast<const float4*>(&As[i][4 * ty]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[i][4 * tx]);
      const float ar[4] = {a.x, a.y, a.z, a.w}, br[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(ar[r], br[q], acc[r][q]);
    }
  }
}

__device__ __forceinline__ void load_tile(const float* src, size_t bh, int d_k, int d_v, int k0, int v0,
                                          float (&x)[4][4]) {
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int row = k0 + 4 * ty + r, col = v0 + 4 * tx + q;
      x[r][q] = src && row < d_k && col < d_v ? src[(bh * d_k + row) * static_cast<size_t>(d_v) + col] : 0.f;
    }
}

// Forward walk: S_{−1} = S_in; S_c = γ^{b_c}·S_{c−1} + Σ_i γ^{b_c−1−i} k′_iᵀ v_i,
// stored for c = 0 … C−1.
template <typename Tin>
__global__ void __launch_bounds__(256) state_walk_fwd_kernel(WalkArgs w) {
  __shared__ __align__(16) float As[kStage][kTile + 4];
  __shared__ __align__(16) float Bs[kStage][kTile + 4];
  const int ntiles = w.ntk * w.ntv;
  const size_t bh = blockIdx.x / ntiles;
  const int tile = blockIdx.x % ntiles;
  const int h = static_cast<int>(bh % w.H);
  const int k0 = (tile / w.ntv) * kTile, v0 = (tile % w.ntv) * kTile;
  float S[4][4];
  load_tile(w.s0, bh, w.d_k, w.d_v, k0, v0, S);
  for (int c = 0; c < w.C; ++c) {
    const int bc = min(kGradChunk, w.L - c * kGradChunk);
    const float g = exp2f(static_cast<float>(bc) * w.cc.lg2g[h]);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) S[r][q] *= g;
    chunk_update<Tin, true>(w, bh, h, c, k0, v0, S, As, Bs);
    float4* dst = reinterpret_cast<float4*>(w.states + ((bh * w.C + c) * ntiles + tile) * 4096) + threadIdx.x * 4;
#pragma unroll
    for (int r = 0; r < 4; ++r) dst[r] = make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
  }
}

// Backward walk: dS_{C−1} = dS_out; dS_{c−1} = γ^{b_c}·dS_c + Σ_j γ^{j+1} q′_jᵀ dO_j.
// At every boundary c = C−1 … −1 it adds the weighted <S_c, dS_c> and Z_c of
// its tile (weights of the boundary split above).
template <typename Tin>
__global__ void __launch_bounds__(256) state_walk_bwd_kernel(WalkArgs w) {
  __shared__ __align__(16) float As[kStage][kTile + 4];
  __shared__ __align__(16) float Bs[kStage][kTile + 4];
  __shared__ float zred[16][2][16];
  __shared__ double gred[256];
  const int ntiles = w.ntk * w.ntv;
  const size_t bh = blockIdx.x / ntiles;
  const int tile = blockIdx.x % ntiles;
  const int h = static_cast<int>(bh % w.H);
  const int k0 = (tile / w.ntv) * kTile, v0 = (tile % w.ntv) * kTile;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int r_last = w.L - (w.C - 1) * kGradChunk;
  float dS[4][4];
  load_tile(w.s0, bh, w.d_k, w.d_v, k0, v0, dS);
  double gacc = 0.0, zacc0 = 0.0, zacc1 = 0.0;
  // boundary products of dS (already dS_c) with S_c
  auto boundary = [&](int c) {
    float Sx[4][4];
    if (c >= 0) {
      const float4* src = reinterpret_cast<const float4*>(w.states + ((bh * w.C + c) * ntiles + tile) * 4096) +
                          threadIdx.x * 4;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 x = src[r];
        Sx[r][0] = x.x; Sx[r][1] = x.y; Sx[r][2] = x.z; Sx[r][3] = x.w;
      }
    } else {
      load_tile(w.s_in, bh, w.d_k, w.d_v, k0, v0, Sx);
    }
    float ip = 0.f, z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int r = 0; r < 4; ++r) ip = fmaf(Sx[r][q], dS[r][q], ip);
      z0 += Sx[1][q] * dS[0][q] - Sx[0][q] * dS[1][q];
      z1 += Sx[3][q] * dS[2][q] - Sx[2][q] * dS[3][q];
    }
    float wg, wt;
    if (c == w.C - 1) {          // checked first: with one chunk, boundary 0 is the last
      wg = static_cast<float>(r_last - 1) - kKappa;
      wt = -(w.pos0 + static_cast<float>((w.C - 1) * kGradChunk) + kKappa);
    } else if (c < 0) {
      wg = 1.f + kKappa;
      wt = w.pos0 + kKappa;
    } else {
      wg = wt = static_cast<float>(kGradChunk);
    }
    gacc += static_cast<double>(wg) * ip;
    zacc0 += static_cast<double>(wt) * z0;
    zacc1 += static_cast<double>(wt) * z1;
  };
  boundary(w.C - 1);
  for (int c = w.C - 1; c >= 0; --c) {
    const int bc = min(kGradChunk, w.L - c * kGradChunk);
    const float g = exp2f(static_cast<float>(bc) * w.cc.lg2g[h]);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) dS[r][q] *= g;
    chunk_update<Tin, false>(w, bh, h, c, k0, v0, dS, As, Bs);   // now dS_{c−1}
    boundary(c - 1);
  }
  // block sums: Σ over threads of gacc; per pair of the tile Σ over tx
  gred[threadIdx.x] = gacc;
  zred[ty][0][tx] = static_cast<float>(zacc0);
  zred[ty][1][tx] = static_cast<float>(zacc1);
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (static_cast<int>(threadIdx.x) < s) gred[threadIdx.x] += gred[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) w.gpart[blockIdx.x] = gred[0];
  if (threadIdx.x < 32) {   // pair p of the tile = 2·ty + u
    const int p = threadIdx.x, yy = p >> 1, u = p & 1;
    float z = 0.f;
    for (int x = 0; x < 16; ++x) z += zred[yy][u][x];
    w.zpart[static_cast<size_t>(blockIdx.x) * 32 + p] = z;
  }
}

// ---------------------------------------------------------------------------
// Faster walks for d_k and d_v multiples of 64.  A prep pass writes the walks'
// left operands once, in fp32: kf[bh][t] = d_k^{-1/2}·γ^{b_c−1−j}·R k_t and
// qb[bh][t] = γ^{j+1}·R q_t.  A walk block (64 threads, one 64 × 64 state
// tile, thread (ty, tx) = (tid / 8, tid % 8) owning rows 8ty … 8ty+7 and
// columns 8tx … 8tx+7) streams the rows of its chunks in stages of 32 through
// a double-buffered shared-memory ring filled by asynchronous copies, so the
// next stage loads while the current one is multiplied.  States are stored
// per (b, h, chunk, tile) as [16 float4 slots][64 threads].
// ---------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(256) walk_prep_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                        float* __restrict__ qb, float* __restrict__ kf,
                                                        const float2* __restrict__ cs, CallConsts cc,
                                                        int H, int L, int d_k, size_t rows) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;   // (row, 4 pairs)
  const int groups = d_k / 8;
  if (idx >= rows * groups) return;
  const size_t row = idx / groups;
  const int g = static_cast<int>(idx % groups);
  const int t = static_cast<int>(row % L);
  const int h = static_cast<int>((row / L) % H);
  const int c = t / kGradChunk, j = t % kGradChunk;
  const int bc = min(kGradChunk, L - c * kGradChunk);
  const float wk = cc.kscale * exp2f(static_cast<float>(bc - 1 - j) * cc.lg2g[h]);
  const float wq = exp2f(static_cast<float>(j + 1) * cc.lg2g[h]);
  float xq[8], xk[8];
  load8(q + row * d_k + 8 * g, xq);
  load8(k + row * d_k + 8 * g, xk);
  float oq[8], ok[8];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 e = cs[static_cast<size_t>(t) * (d_k / 2) + 4 * g + u];
    oq[2 * u] = wq * fmaf(xq[2 * u], e.x, -xq[2 * u + 1] * e.y);
    oq[2 * u + 1] = wq * fmaf(xq[2 * u + 1], e.x, xq[2 * u] * e.y);
    ok[2 * u] = wk * fmaf(xk[2 * u], e.x, -xk[2 * u + 1] * e.y);
    ok[2 * u + 1] = wk * fmaf(xk[2 * u + 1], e.x, xk[2 * u] * e.y);
  }
  store8(qb + row * d_k + 8 * g, oq);
  store8(kf + row * d_k + 8 * g, ok);
}

template <typename Tin>
struct Walk2Smem {
  static constexpr int A_BYTES = kStage * kTile * 4;
  static constexpr int B_BYTES = kStage * kTile * static_cast<int>(sizeof(Tin));
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int BYTES = 2 * STAGE;
};

// Stage s of a walk: rows [t0, t0 + n) of the sequence (n ≤ 32, all in one chunk).
struct StageRows { int c, t0, n; };

__device__ __forceinline__ StageRows walk_stage(int s, int L, int C, bool fwd) {
  StageRows r;
  if (fwd) {
    r.t0 = kStage * s;
    r.c = r.t0 / kGradChunk;
  } else {   // chunks from the last down, rows ascending inside each
    const int rl = L - (C - 1) * kGradChunk;
    const int nl = (rl + kStage - 1) / kStage;
    if (s < nl) {
      r.c = C - 1;
      r.t0 = (C - 1) * kGradChunk + kStage * s;
    } else {
      const int s2 = s - nl;
      r.c = C - 2 - s2 / (kGradChunk / kStage);
      r.t0 = r.c * kGradChunk + kStage * (s2 % (kGradChunk / kStage));
    }
  }
  r.n = min(kStage, min(L, (r.c + 1) * kGradChunk) - r.t0);
  return r;
}

template <typename Tin, bool FWD>
__global__ void __launch_bounds__(64) state_walk2_kernel(WalkArgs w, const float* __restrict__ aop) {
  extern __shared__ __align__(16) unsigned char wsm[];
  using SM = Walk2Smem<Tin>;
  constexpr int PER = 16 / sizeof(Tin);
  const int ntiles = w.ntk * w.ntv;
  const size_t bh = blockIdx.x / ntiles;
  const int tile = blockIdx.x % ntiles;
  const int h = static_cast<int>(bh % w.H);
  const int k0 = (tile / w.ntv) * kTile, v0 = (tile % w.ntv) * kTile;
  const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;
  const Tin* Bm = static_cast<const Tin*>(w.b);
  const int rl = w.L - (w.C - 1) * kGradChunk;
  const int nstages = (w.C - 1) * (kGradChunk / kStage) + (rl + kStage - 1) / kStage;

  auto issue = [&](int s) {
    if (s < nstages) {
      const StageRows sr = walk_stage(s, w.L, w.C, FWD);
      float* As = reinterpret_cast<float*>(wsm + (s & 1) * SM::STAGE);
      Tin* Bs = reinterpret_cast<Tin*>(wsm + (s & 1) * SM::STAGE + SM::A_BYTES);
      for (int e = tid; e < sr.n * (kTile / 4); e += 64) {     // A: 16 pieces per row
        const int r = e / (kTile / 4), pc = e % (kTile / 4);
        cp_async16(As + r * kTile + 4 * pc, aop + (bh * w.L + sr.t0 + r) * static_cast<size_t>(w.d_k) + k0 + 4 * pc);
      }
      constexpr int BP = kTile / PER;                          // B pieces per row
      for (int e = tid; e < sr.n * BP; e += 64) {
        const int r = e / BP, pc = e % BP;
        cp_async16(Bs + r * kTile + PER * pc, Bm + (bh * w.L + sr.t0 + r) * static_cast<size_t>(w.d_v) + v0 + PER * pc);
      }
    }
    cp_async_commit();
  };

  float acc[8][8];
  {   // S_in (forward) or dS_out (backward)
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int q = 0; q < 8; ++q)
        acc[r][q] = w.s0 ? w.s0[(bh * w.d_k + k0 + 8 * ty + r) * static_cast<size_t>(w.d_v) + v0 + 8 * tx + q] : 0.f;
  }
  double gacc = 0.0, zacc[4] = {0.0, 0.0, 0.0, 0.0};
  auto state_slot = [&](int c) {
    return reinterpret_cast<float4*>(w.states + ((bh * w.C + c) * ntiles + tile) * 4096);
  };
  // backward: weighted boundary products of acc (= dS_c) with S_c
  auto boundary = [&](int c) {
    float ip = 0.f, z[4] = {0.f, 0.f, 0.f, 0.f};
    const float4* src = c >= 0 ? state_slot(c) : nullptr;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float sx[8];
      if (c >= 0) {
        const float4 a = src[(2 * r) * 64 + tid], b = src[(2 * r + 1) * 64 + tid];
        sx[0] = a.x; sx[1] = a.y; sx[2] = a.z; sx[3] = a.w; sx[4] = b.x; sx[5] = b.y; sx[6] = b.z; sx[7] = b.w;
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          sx[q] = w.s_in ? w.s_in[(bh * w.d_k + k0 + 8 * ty + r) * static_cast<size_t>(w.d_v) + v0 + 8 * tx + q] : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) ip = fmaf(sx[q], acc[r][q], ip);
      if (r & 1) {   // pair (r − 1, r): Σ S[r]·dS[r−1] − S[r−1]·dS[r]; S[r−1] kept from the last row
#pragma unroll
        for (int q = 0; q < 8; ++q) z[r >> 1] += sx[q] * acc[r - 1][q];
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) z[r >> 1] -= sx[q] * acc[r + 1][q];
      }
    }
    float wg, wt;
    if (c == w.C - 1) {
      wg = static_cast<float>(rl - 1) - kKappa;
      wt = -(w.pos0 + static_cast<float>((w.C - 1) * kGradChunk) + kKappa);
    } else if (c < 0) {
      wg = 1.f + kKappa;
      wt = w.pos0 + kKappa;
    } else {
      wg = wt = static_cast<float>(kGradChunk);
    }
    gacc += static_cast<double>(wg) * ip;
#pragma unroll
    for (int p = 0; p < 4; ++p) zacc[p] += static_cast<double>(wt) * z[p];
  };
  if (!FWD) boundary(w.C - 1);

  issue(0);
  for (int s = 0; s < nstages; ++s) {
    const StageRows sr = walk_stage(s, w.L, w.C, FWD);
    const int bc = min(kGradChunk, w.L - sr.c * kGradChunk);
    if (sr.t0 == sr.c * kGradChunk) {   // first stage of a chunk: decay the carried state
      const float g = exp2f(static_cast<float>(bc) * w.cc.lg2g[h]);
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[r][q] *= g;
    }
    issue(s + 1);
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    const float* As = reinterpret_cast<const float*>(wsm + (s & 1) * SM::STAGE);
    const Tin* Bs = reinterpret_cast<const Tin*>(wsm + (s & 1) * SM::STAGE + SM::A_BYTES);
    auto step = [&](int i) {
      const float4 a0 = *reinterpret_cast<const float4*>(As + i * kTile + 8 * ty);
      const float4 a1 = *reinterpret_cast<const float4*>(As + i * kTile + 8 * ty + 4);
      float bv[8];
      lds8(Bs + i * kTile + 8 * tx, bv);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[r][q] = fmaf(av[r], bv[q], acc[r][q]);
    };
    if (sr.n == kStage) {   // full stage: unrolled, so the next rows' loads issue early
#pragma unroll 8
      for (int i = 0; i < kStage; ++i) step(i);
    } else {
      for (int i = 0; i < sr.n; ++i) step(i);
    }
    __syncthreads();   // the buffer of stage s is refilled by issue(s + 2)
    if (sr.t0 + sr.n == sr.c * kGradChunk + bc) {   // last stage of the chunk
      if (FWD) {
        float4* dst = state_slot(sr.c);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          dst[(2 * r) * 64 + tid] = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
          dst[(2 * r + 1) * 64 + tid] = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
        }
      } else {
        boundary(sr.c - 1);
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (FWD) return;
  __shared__ double gred[64];
  __shared__ float zred[8][4][8];
  gred[tid] = gacc;
#pragma unroll
  for (int p = 0; p < 4; ++p) zred[ty][p][tx] = static_cast<float>(zacc[p]);
  __syncthreads();
  if (tid == 0) {
    double t = 0.0;
    for (int i = 0; i < 64; ++i) t += gred[i];
    w.gpart[blockIdx.x] = t;
  }
  if (tid < 32) {   // tile pair 4·ty + p = rows 8ty + 2p, 8ty + 2p + 1
    const int yy = tid >> 2, p = tid & 3;
    float z = 0.f;
    for (int x = 0; x < 8; ++x) z += zred[yy][p][x];
    w.zpart[static_cast<size_t>(blockIdx.x) * 32 + tid] = z;
  }
}

// Finishing sums, in double and in a fixed order (strided per thread, then a
// fixed tree).  Blocks [0, H): dγ_h = γ_h⁻¹ · (the B·nseg row partials +
// the B·tiles boundary partials of head h).  Blocks [H, H + P): dθ_i = the
// B·H·nseg row partials of pair i + the B·H·ntv boundary partials of its tile.
struct FinishArgs {
  const double* gpart; const double* gwalk; const float* tpart; const float* zpart;
  float* d_gamma; float* d_theta;
  int B, H, nseg, P, ntk, ntv;
  double inv_gamma[kMaxHeads];
};

__device__ __forceinline__ double block_sum_256(double s, double* red) {
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  return red[0];
}

__global__ void __launch_bounds__(256) param_finish_kernel(FinishArgs a) {
  __shared__ double red[256];
  const int ntiles = a.ntk * a.ntv;
  if (static_cast<int>(blockIdx.x) < a.H) {
    if (!a.d_gamma) return;
    const int h = blockIdx.x;
    double s = 0.0;
    for (int i = threadIdx.x; i < a.B * a.nseg; i += 256) {
      const int b = i / a.nseg, seg = i % a.nseg;
      s += a.gpart[(static_cast<size_t>(b) * a.H + h) * a.nseg + seg];
    }
    for (int i = threadIdx.x; i < a.B * ntiles; i += 256) {
      const int b = i / ntiles, tl = i % ntiles;
      s += a.gwalk[(static_cast<size_t>(b) * a.H + h) * ntiles + tl];
    }
    s = block_sum_256(s, red);
    if (threadIdx.x == 0) a.d_gamma[h] = static_cast<float>(s * a.inv_gamma[h]);
    return;
  }
  if (!a.d_theta) return;
  const int i = blockIdx.x - a.H;
  const size_t nblk = static_cast<size_t>(a.B) * a.H * a.nseg;
  const float* src = a.tpart + static_cast<size_t>(i) * nblk;
  double s = 0.0;
  for (size_t blk = threadIdx.x; blk < nblk; blk += 256) s += src[blk];
  const int tk = i / 32, pl = i % 32;
  const size_t nwalk = static_cast<size_t>(a.B) * a.H * a.ntv;
  for (size_t m = threadIdx.x; m < nwalk; m += 256) {
    const size_t bh = m / a.ntv;
    const int tv = static_cast<int>(m % a.ntv);
    s += a.zpart[((bh * ntiles) + static_cast<size_t>(tk) * a.ntv + tv) * 32 + pl];
  }
  s = block_sum_256(s, red);
  if (threadIdx.x == 0) a.d_theta[i] = static_cast<float>(s);
}

// ---------------------------------------------------------------------------
// GroupNorm backward.  Block = (b, h, segment of kRowsPerBlock tokens),
// 4 warps, one row per warp at a time (the row stays in registers: NV
// channels per lane, d_v ≤ 32·NV, NV ∈ {8, 16, 32}).  dx written per row; the segment's
// Σ dy ⊙ x̂ and Σ dy per channel go to wpart[block][2][d_v] (null: not
// wanted).  VEC: d_v a multiple of 8 (lane owns channels 8·(lane + 32j) … +7),
// otherwise lane owns channels lane + 32j.
// ---------------------------------------------------------------------------
template <typename Tx, typename Tg, bool VEC, int NV>
__global__ void __launch_bounds__(128) gn_backward_kernel(const Tx* __restrict__ x,
                                                          const Tx* __restrict__ dy,
                                                          const float* __restrict__ w,
                                                          Tg* __restrict__ dx,
                                                          float* __restrict__ wpart, int H, int L,
                                                          int d_v, int nseg, float eps) {
  extern __shared__ float wsum[];   // [4 warps][2][d_v] when wpart is set
  constexpr int R = NV >= 32 ? 1 : 2;   // rows in flight per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x % nseg;
  const size_t bh = blockIdx.x / nseg;
  const int h = static_cast<int>(bh % H);
  const int t0 = seg * kRowsPerBlock, t1 = min(L, t0 + kRowsPerBlock);
  const float inv_n = 1.f / static_cast<float>(d_v);
  auto chan = [&](int e) {   // channel of this lane's e-th value (−1: none)
    const int c = VEC ? 8 * (lane + 32 * (e >> 3)) + (e & 7) : lane + 32 * e;
    return c < d_v ? c : -1;
  };
  float aw[NV], ab[NV], wv[NV];
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    aw[e] = ab[e] = 0.f;
    const int c = chan(e);
    wv[e] = c < 0 ? 0.f : (w ? __ldg(w + static_cast<size_t>(h) * d_v + c) : 1.f);
  }

  for (int t = t0 + warp; t < t1; t += 4 * R) {
    float xv[R][NV], gv[R][NV];
    bool live[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {   // all loads of the R rows first
      const int tr = t + 4 * r;
      live[r] = tr < t1;
      const size_t row = bh * L + (live[r] ? tr : t);
      const Tx* xr = x + row * d_v;
      const Tx* gr = dy + row * d_v;
#pragma unroll
      for (int j = 0; j < NV / 8; ++j) {
        if (VEC) {
          const int c = 8 * (lane + 32 * j);
          float a8[8], b8[8];
          if (c < d_v) {
            load8(xr + c, a8);
            load8(gr + c, b8);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) a8[e] = b8[e] = 0.f;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) { xv[r][8 * j + e] = a8[e]; gv[r][8 * j + e] = b8[e]; }
        } else {
#pragma unroll
          for (int e = 8 * j; e < 8 * j + 8; ++e) {
            const int c = lane + 32 * e;
            xv[r][e] = c < d_v ? to_f32(xr[c]) : 0.f;
            gv[r][e] = c < d_v ? to_f32(gr[c]) : 0.f;
          }
        }
      }
    }
    float mu[R], rstd[R], mg[R], mgx[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < NV; ++e) s += xv[r][e];
      mu[r] = warp_sum(s) * inv_n;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float q = 0.f;
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const float d = chan(e) >= 0 ? xv[r][e] - mu[r] : 0.f;
        q = fmaf(d, d, q);
      }
      rstd[r] = rsqrtf(warp_sum(q) * inv_n + eps);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float sg = 0.f, sgx = 0.f;
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const float xh = chan(e) >= 0 ? (xv[r][e] - mu[r]) * rstd[r] : 0.f;
        const float gw = gv[r][e] * wv[e];
        if (live[r]) {
          aw[e] = fmaf(gv[r][e], xh, aw[e]);
          ab[e] += gv[r][e];
        }
        xv[r][e] = xh;
        gv[r][e] = gw;
        sg += gw;
        sgx = fmaf(gw, xh, sgx);
      }
      mg[r] = warp_sum(sg) * inv_n;
      mgx[r] = warp_sum(sgx) * inv_n;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (!live[r]) continue;
      Tg* dr = dx + (bh * L + t + 4 * r) * d_v;
#pragma unroll
      for (int j = 0; j < NV / 8; ++j) {
        if (VEC) {
          const int c = 8 * (lane + 32 * j);
          if (c < d_v) {
            float o8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o8[e] = rstd[r] * (gv[r][8 * j + e] - mg[r] - xv[r][8 * j + e] * mgx[r]);
            store8(dr + c, o8);
          }
        } else {
#pragma unroll
          for (int e = 8 * j; e < 8 * j + 8; ++e) {
            const int c = lane + 32 * e;
            if (c < d_v) dr[c] = from_f32<Tg>(rstd[r] * (gv[r][e] - mg[r] - xv[r][e] * mgx[r]));
          }
        }
      }
    }
  }
  if (!wpart) return;
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    const int c = chan(e);
    if (c >= 0) {
      wsum[(warp * 2) * d_v + c] = aw[e];
      wsum[(warp * 2 + 1) * d_v + c] = ab[e];
    }
  }
  __syncthreads();
  float* dst = wpart + static_cast<size_t>(blockIdx.x) * 2 * d_v;
  for (int c = threadIdx.x; c < d_v; c += 128) {
    float sw = 0.f, sb = 0.f;
#pragma unroll
    for (int w4 = 0; w4 < 4; ++w4) {
      sw += wsum[(w4 * 2) * d_v + c];
      sb += wsum[(w4 * 2 + 1) * d_v + c];
    }
    dst[c] = sw;
    dst[d_v + c] = sb;
  }
}

// The same computation for 16-byte rows (d_v a multiple of 8), with the rows
// staged through shared memory by per-lane asynchronous copies: each lane
// copies the 16-byte pieces of x and dy it owns (channels 8·(lane + 32j) …
// +7) for the next R rows while it works on the current R rows from the
// other stage, so loads stay in flight during the reductions.  A lane only
// ever reads the pieces it copied itself, so its own wait_group is the only
// synchronisation.  Shared memory: [4 warps][2 stages][R][x, dy][d_v] plus,
// after the loop, the [4 warps][2][d_v] parameter sums in the same space.
template <typename Tx, typename Tg, int NV>
__global__ void __launch_bounds__(128) gn_backward_async_kernel(const Tx* __restrict__ x,
                                                                const Tx* __restrict__ dy,
                                                                const float* __restrict__ w,
                                                                Tg* __restrict__ dx,
                                                                float* __restrict__ wpart, int H,
                                                                int L, int d_v, int nseg, float eps) {
  extern __shared__ __align__(16) unsigned char gsm[];
  constexpr int R = 2;                       // rows per stage and warp
  constexpr int PER = 16 / sizeof(Tx);       // elements per 16-byte piece (8 or 4)
  constexpr int NP = NV / 8;                 // 8-channel groups per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x % nseg;
  const size_t bh = blockIdx.x / nseg;
  const int h = static_cast<int>(bh % H);
  const int t0 = seg * kRowsPerBlock, t1 = min(L, t0 + kRowsPerBlock);
  const float inv_n = 1.f / static_cast<float>(d_v);
  Tx* stage = reinterpret_cast<Tx*>(gsm) + static_cast<size_t>(warp) * 2 * R * 2 * d_v;
  auto buf = [&](int st, int r, int arr) { return stage + ((st * R + r) * 2 + arr) * static_cast<size_t>(d_v); };
  // issue the copies of the R rows starting at token tt into stage st
  auto issue = [&](int tt, int st) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int tr = tt + 4 * r;
      if (tr >= t1) continue;
      const size_t row = (bh * L + tr) * static_cast<size_t>(d_v);
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        const int c = 8 * (lane + 32 * j);
        if (c >= d_v) continue;
#pragma unroll
        for (int u = 0; u < 8; u += PER) {
          cp_async16(buf(st, r, 0) + c + u, x + row + c + u);
          cp_async16(buf(st, r, 1) + c + u, dy + row + c + u);
        }
      }
    }
    cp_async_commit();
  };
  float aw[NV], ab[NV], wv[NV];
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    aw[e] = ab[e] = 0.f;
    const int c = 8 * (lane + 32 * (e >> 3)) + (e & 7);
    wv[e] = c >= d_v ? 0.f : (w ? __ldg(w + static_cast<size_t>(h) * d_v + c) : 1.f);
  }
  int st = 0;
  issue(t0 + warp, 0);
  for (int t = t0 + warp; t < t1; t += 4 * R, st ^= 1) {
    issue(t + 4 * R, st ^ 1);   // the next rows (an empty group past the end)
    cp_async_wait1();           // this lane's copies of the current rows have landed
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int tr = t + 4 * r;
      if (tr >= t1) break;      // uniform across the warp
      float xv[NV], gv[NV];
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        const int c = 8 * (lane + 32 * j);
        float a8[8], b8[8];
        if (c < d_v) {
          lds8(buf(st, r, 0) + c, a8);
          lds8(buf(st, r, 1) + c, b8);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) a8[e] = b8[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) { xv[8 * j + e] = a8[e]; gv[8 * j + e] = b8[e]; }
      }
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < NV; ++e) s += xv[e];
      const float mu = warp_sum(s) * inv_n;
      float q = 0.f;
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const int c = 8 * (lane + 32 * (e >> 3)) + (e & 7);
        const float d = c < d_v ? xv[e] - mu : 0.f;
        q = fmaf(d, d, q);
      }
      const float rstd = rsqrtf(warp_sum(q) * inv_n + eps);
      float sg = 0.f, sgx = 0.f;
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const int c = 8 * (lane + 32 * (e >> 3)) + (e & 7);
        const float xh = c < d_v ? (xv[e] - mu) * rstd : 0.f;
        const float gw = gv[e] * wv[e];
        aw[e] = fmaf(gv[e], xh, aw[e]);
        ab[e] += gv[e];
        xv[e] = xh;
        gv[e] = gw;
        sg += gw;
        sgx = fmaf(gw, xh, sgx);
      }
      const float mg = warp_sum(sg) * inv_n, mgx = warp_sum(sgx) * inv_n;
      Tg* dr = dx + (bh * L + tr) * static_cast<size_t>(d_v);
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        const int c = 8 * (lane + 32 * j);
        if (c < d_v) {
          float o8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o8[e] = rstd * (gv[8 * j + e] - mg - xv[8 * j + e] * mgx);
          store8(dr + c, o8);
        }
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (!wpart) return;
  __syncthreads();   // every warp is done with the stages: reuse them for the sums
  float* wsum = reinterpret_cast<float*>(gsm);
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    const int c = 8 * (lane + 32 * (e >> 3)) + (e & 7);
    if (c < d_v) {
      wsum[(warp * 2) * d_v + c] = aw[e];
      wsum[(warp * 2 + 1) * d_v + c] = ab[e];
    }
  }
  __syncthreads();
  float* dst = wpart + static_cast<size_t>(blockIdx.x) * 2 * d_v;
  for (int c = threadIdx.x; c < d_v; c += 128) {
    float sw = 0.f, sb = 0.f;
#pragma unroll
    for (int w4 = 0; w4 < 4; ++w4) {
      sw += wsum[(w4 * 2) * d_v + c];
      sb += wsum[(w4 * 2 + 1) * d_v + c];
    }
    dst[c] = sw;
    dst[d_v + c] = sb;
  }
}

// GroupNorm forward over 16-byte rows (d_v a multiple of 8): one group per
// (b, h, t) row over its d_v channels, biased variance (mean first, then the
// centred sum of squares), optional affine («从RoPE到Retention…» §5).  The
// rows are held in registers as raw 16-byte vectors (converted to fp32 at
// each use, so that a warp keeps 8 KB of loads in flight in 32 registers a
// lane): a warp takes RW rows at a time with all their loads issued before
// any arithmetic, grid-stride over the row groups.  y may be x (same type):
// a lane writes only the channels it read itself.  w, b 16-byte aligned
// (checked by the callers).
template <typename Tx>
__device__ __forceinline__ void unpack8(const uint4* v, float (&o)[8]) {
  if constexpr (sizeof(Tx) == 2) {
    const uint32_t wd[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = bf16lo_to_f32(wd[i]);
      o[2 * i + 1] = bf16hi_to_f32(wd[i]);
    }
  } else {
    o[0] = __uint_as_float(v[0].x); o[1] = __uint_as_float(v[0].y);
    o[2] = __uint_as_float(v[0].z); o[3] = __uint_as_float(v[0].w);
    o[4] = __uint_as_float(v[1].x); o[5] = __uint_as_float(v[1].y);
    o[6] = __uint_as_float(v[1].z); o[7] = __uint_as_float(v[1].w);
  }
}

template <typename Tx, typename Ty, int NV>
__global__ void __launch_bounds__(256, 3) gn_forward_reg_kernel(const Tx* x, Ty* y,
                                                                const float* __restrict__ w,
                                                                const float* __restrict__ b, int H,
                                                                int L, int d_v, size_t rows, float eps) {
  constexpr int NP = NV / 8;                          // 8-channel pieces per lane
  constexpr int U4 = 8 * static_cast<int>(sizeof(Tx)) / 16;   // 16-byte vectors per piece
  constexpr int RW = (8 / (NP * U4)) > 0 ? 8 / (NP * U4) : 1;
  const int lane = threadIdx.x & 31;
  const size_t wg = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const size_t nw = (static_cast<size_t>(gridDim.x) * blockDim.x) >> 5;
  const float inv_n = 1.f / static_cast<float>(d_v);
  for (size_t r0 = wg * RW; r0 < rows; r0 += nw * RW) {
    uint4 raw[RW][NP][U4];
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        const int c = 8 * (lane + 32 * j);
#pragma unroll
        for (int u = 0; u < U4; ++u)
          raw[r][j][u] = (r0 + r < rows && c < d_v)
                             ? *reinterpret_cast<const uint4*>(x + (r0 + r) * d_v + c + u * (16 / sizeof(Tx)))
                             : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      const size_t row = r0 + r;
      if (row >= rows) break;
      const int h = static_cast<int>((row / L) % H);
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        float f[8];
        unpack8<Tx>(raw[r][j], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += f[e];
      }
      const float mu = warp_sum(s) * inv_n;
      float q = 0.f;
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        float f[8];
        unpack8<Tx>(raw[r][j], f);
        const bool live = 8 * (lane + 32 * j) < d_v;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float d = live ? f[e] - mu : 0.f;
          q = fmaf(d, d, q);
        }
      }
      const float rstd = rsqrtf(warp_sum(q) * inv_n + eps);
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        const int c = 8 * (lane + 32 * j);
        if (c >= d_v) continue;
        float f[8], o8[8];
        unpack8<Tx>(raw[r][j], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) o8[e] = (f[e] - mu) * rstd;
        if (w) {
          const float4 u0 = __ldg(reinterpret_cast<const float4*>(w + static_cast<size_t>(h) * d_v + c));
          const float4 u1 = __ldg(reinterpret_cast<const float4*>(w + static_cast<size_t>(h) * d_v + c) + 1);
          o8[0] *= u0.x; o8[1] *= u0.y; o8[2] *= u0.z; o8[3] *= u0.w;
          o8[4] *= u1.x; o8[5] *= u1.y; o8[6] *= u1.z; o8[7] *= u1.w;
        }
        if (b) {
          const float4 u0 = __ldg(reinterpret_cast<const float4*>(b + static_cast<size_t>(h) * d_v + c));
          const float4 u1 = __ldg(reinterpret_cast<const float4*>(b + static_cast<size_t>(h) * d_v + c) + 1);
          o8[0] += u0.x; o8[1] += u0.y; o8[2] += u0.z; o8[3] += u0.w;
          o8[4] += u1.x; o8[5] += u1.y; o8[6] += u1.z; o8[7] += u1.w;
        }
        store8(y + row * d_v + c, o8);
      }
    }
  }
}

// d_weight[h][c], d_bias[h][c] = Σ over b and segments of wpart, in double.
// grid = (⌈d_v/32⌉, H), block = 32 channels × 8 row groups; group r takes the
// partials r, r + 8, … and the 8 group sums are added in order.
__global__ void __launch_bounds__(256) gn_param_finish_kernel(const float* __restrict__ wpart,
                                                              float* d_weight, float* d_bias,
                                                              int B, int H, int d_v, int nseg) {
  __shared__ double red[2][8][32];
  const int cx = threadIdx.x & 31, r = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + cx;
  const int h = blockIdx.y;
  double sw = 0.0, sb = 0.0;
  if (c < d_v) {
    const int n = B * nseg;
    for (int i0 = r; i0 < n; i0 += 64) {   // eight partials of this group in flight
      float fw[8], fb[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + 8 * u;
        fw[u] = fb[u] = 0.f;
        if (i < n) {
          const int b = i / nseg, seg = i % nseg;
          const float* p = wpart + ((static_cast<size_t>(b) * H + h) * nseg + seg) * 2 * d_v;
          fw[u] = p[c];
          fb[u] = p[d_v + c];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) { sw += fw[u]; sb += fb[u]; }
    }
  }
  red[0][r][cx] = sw;
  red[1][r][cx] = sb;
  __syncthreads();
  if (r == 0 && c < d_v) {
    double tw = 0.0, tb = 0.0;
    for (int g = 0; g < 8; ++g) { tw += red[0][g][cx]; tb += red[1][g][cx]; }
    if (d_weight) d_weight[static_cast<size_t>(h) * d_v + c] = static_cast<float>(tw);
    if (d_bias) d_bias[static_cast<size_t>(h) * d_v + c] = static_cast<float>(tb);
  }
}

}  // namespace grad
}  // namespace ret
