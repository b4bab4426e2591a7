// Parameter gradients of the retention core (γ per head, θ per rotation
// pair) and the GroupNorm backward.  All HBM-bound row passes.
//
// dγ_h.  Differentiating the decay factors of the parallel form with its
// state terms («从RoPE到Retention…» §3 and §4.1; ∂γ^e/∂γ = e·γ^{e−1})
// gives γ⁻¹·Σ (n − m)·A_nm over every (query n, key m) pair, A_nm being the
// pair's share of <dO, out> + <dS_out, S_out>.  The row sums of A are
// dO_n·o_n (the state_in term counted as a key at m = −1, the state_out read
// as a query at n = L − 1) and its column sums are v_m·dv_m, so per (b, h)
//   γ·dγ = Σ_t t·(dO_t·o_t − v_t·dv_t) + <S_in, dS_in> + (L − 1)·<dS_out, S_out>
// with t the local token index (the decay depends on index differences only).
//
// dθ_i.  Pair i of q′_t is pair i of q_t rotated by (pos0 + t)·θ_i («从RoPE到
// Retention…» §2, where θ is learnable), so ∂q′/∂θ_i = (pos0 + t)·J q′ on that
// pair, J(a, b) = (−b, a).  With dq = Rᵀ dQ′ and J commuting with the
// rotation, dQ′·J q′ = dq·J q, and likewise for k (the 1/√d_k scale cancels
// between dk and k′):
//   dθ_i = Σ_{b,h,t} (pos0 + t)·(dq₂ᵢ₊₁ q₂ᵢ − dq₂ᵢ q₂ᵢ₊₁ + dk₂ᵢ₊₁ k₂ᵢ − dk₂ᵢ k₂ᵢ₊₁)
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

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// ---------------------------------------------------------------------------
// Row pass of the parameter gradients.  Block = (b, h, segment of
// kRowsPerBlock tokens), 8 warps, warp w takes tokens w, w + 8, …  Writes
// gpart[block] (the segment's Σ t·(dO·o − v·dv), double) and tpart[i][block]
// (the segment's share of dθ_i; pair-major, so the finishing sums read it
// contiguously).  VEC: d_k and d_v are multiples of 8 (rows
// read as 16-byte vectors); otherwise element by element.
// ---------------------------------------------------------------------------
struct ParamArgs {
  const void* q; const void* k; const void* v; const void* d_out;
  const void* out; const void* dq; const void* dk; const void* dv;
  int H, L, d_k, d_v, nseg;
  float pos0;          // exact: pos0 + L ≤ 2^24
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
      gacc = fmaf(static_cast<float>(t), s, gacc);
    }
    if (a.tpart) {
      const float pos = a.pos0 + static_cast<float>(t);
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

// <S_in, dS_in> + (L − 1)·<dS_out, S_out> per (b, h), in NS slices:
// spart[bh·NS + slice] (double).  Either product may be absent (null).
constexpr int kStateSlices = 16;

__global__ void __launch_bounds__(256) state_dot_kernel(const float* s_in, const float* ds_in,
                                                        const float* s_out, const float* ds_out,
                                                        int n, float lm1, double* spart) {
  __shared__ double red[8];
  const size_t bh = blockIdx.x / kStateSlices;
  const int slice = blockIdx.x % kStateSlices;
  const int per = (n + kStateSlices - 1) / kStateSlices;
  const int i0 = slice * per, i1 = min(n, i0 + per);
  float s = 0.f;
  const size_t base = bh * static_cast<size_t>(n);
  for (int i = i0 + threadIdx.x; i < i1; i += 256) {
    if (s_in) s = fmaf(s_in[base + i], ds_in[base + i], s);
    if (ds_out) s = fmaf(lm1 * ds_out[base + i], s_out[base + i], s);
  }
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = static_cast<double>(s);
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < 8; ++w) t += red[w];
    spart[blockIdx.x] = t;
  }
}

// Finishing sums, in double and in a fixed order (strided per thread, then a
// fixed tree).  Blocks [0, H): dγ_h over the B·nseg row partials and
// B·kStateSlices state partials of head h, times 1/γ_h.  Blocks [H, H + P):
// dθ_i over the B·H·nseg row partials of pair i.
struct FinishArgs {
  const double* gpart; const double* spart; const float* tpart;
  float* d_gamma; float* d_theta;
  int B, H, nseg, P, have_state;
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
  if (static_cast<int>(blockIdx.x) < a.H) {
    if (!a.d_gamma) return;
    const int h = blockIdx.x;
    double s = 0.0;
    for (int i = threadIdx.x; i < a.B * a.nseg; i += 256) {
      const int b = i / a.nseg, seg = i % a.nseg;
      s += a.gpart[(static_cast<size_t>(b) * a.H + h) * a.nseg + seg];
    }
    if (a.have_state)
      for (int i = threadIdx.x; i < a.B * kStateSlices; i += 256) {
        const int b = i / kStateSlices, sl = i % kStateSlices;
        s += a.spart[(static_cast<size_t>(b) * a.H + h) * kStateSlices + sl];
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
  float aw[NV], ab[NV];
#pragma unroll
  for (int e = 0; e < NV; ++e) aw[e] = ab[e] = 0.f;

  for (int t = t0 + warp; t < t1; t += 4) {
    const size_t row = bh * L + t;
    const Tx* xr = x + row * d_v;
    const Tx* gr = dy + row * d_v;
    float xv[NV], gv[NV];
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
        for (int e = 0; e < 8; ++e) { xv[8 * j + e] = a8[e]; gv[8 * j + e] = b8[e]; }
      } else {
#pragma unroll
        for (int e = 8 * j; e < 8 * j + 8; ++e) {
          const int c = lane + 32 * e;
          xv[e] = c < d_v ? to_f32(xr[c]) : 0.f;
          gv[e] = c < d_v ? to_f32(gr[c]) : 0.f;
        }
      }
    }
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < NV; ++e) s += xv[e];
    const float mu = warp_sum(s) * inv_n;
    float q = 0.f;
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const float d = chan(e) >= 0 ? xv[e] - mu : 0.f;
      q = fmaf(d, d, q);
    }
    const float rstd = rsqrtf(warp_sum(q) * inv_n + eps);
    float sg = 0.f, sgx = 0.f;
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int c = chan(e);
      const float xh = (xv[e] - mu) * rstd;
      const float gw = c >= 0 ? gv[e] * (w ? __ldg(w + static_cast<size_t>(h) * d_v + c) : 1.f) : 0.f;
      aw[e] = fmaf(gv[e], c >= 0 ? xh : 0.f, aw[e]);
      ab[e] += gv[e];
      xv[e] = xh;
      gv[e] = gw;
      sg += gw;
      sgx = fmaf(gw, xh, sgx);
    }
    const float mg = warp_sum(sg) * inv_n, mgx = warp_sum(sgx) * inv_n;
    Tg* dr = dx + row * d_v;
#pragma unroll
    for (int j = 0; j < NV / 8; ++j) {
      if (VEC) {
        const int c = 8 * (lane + 32 * j);
        if (c < d_v) {
          float o8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o8[e] = rstd * (gv[8 * j + e] - mg - xv[8 * j + e] * mgx);
          store8(dr + c, o8);
        }
      } else {
#pragma unroll
        for (int e = 8 * j; e < 8 * j + 8; ++e) {
          const int c = lane + 32 * e;
          if (c < d_v) dr[c] = from_f32<Tg>(rstd * (gv[e] - mg - xv[e] * mgx));
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
  if (c < d_v)
    for (int i = r; i < B * nseg; i += 8) {
      const int b = i / nseg, seg = i % nseg;
      const float* p = wpart + ((static_cast<size_t>(b) * H + h) * nseg + seg) * 2 * d_v;
      sw += p[c];
      sb += p[d_v + c];
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
