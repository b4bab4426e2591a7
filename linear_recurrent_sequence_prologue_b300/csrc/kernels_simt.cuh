// fp32 FFMA kernels: the Θ prologue, the chunk-parallel layout of the
// chunkwise form (per-chunk ΔS, state scan, per-chunk outputs), GroupNorm,
// and the recurrent decode step.
//
// Chunkwise form («从RoPE到Retention…» §4.3; RetNet 保留网络 explainer 分块循环)
// with S the state entering chunk i and j, m local indices in the chunk:
//   o_j   = γ^{j+1} q′_j S + Σ_{m≤j} γ^{j−m} (q′_j·k′_m) v_m
//   ΔS_i  = Σ_j γ^{r−1−j} k′_jᵀ v_j        (r = chunk length)
//   S_i   = fmaf(γ^r, S_{i−1}, ΔS_i)
// The parallel form (§4.1) is the same kernel with one chunk of length L.
#pragma once

#include "common.cuh"

namespace ret {
namespace simt {

// ---------------------------------------------------------------------------
// Θ prologue: y[bh, t, :] = scale · R((pos0 + t)θ) x[bh, t, :]   (§2 theta_shift)
// with pos0 the row's own start when rp.on (row = bh / H).
// flip (for the gradients): bit 0 reads x at row L−1−t, bit 1 writes y at row
// L−1−t; the angle always belongs to position pos0 + t.
// Block (32, 8): x → pair index, y → row.  Angles depend on (position, i)
// only, so each thread loops over the BH heads with one sincos per row start.
// ---------------------------------------------------------------------------
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) rotate_kernel(const Tin* __restrict__ x,
                                                     Tout* __restrict__ y, CallConsts cc,
                                                     int BH, int H, int L, int d, float pos0,
                                                     float scale, RowPos rp, int flip) {
  const int i = blockIdx.x * 32 + threadIdx.x;   // pair
  // row (groups of 8 rows folded over grid.y and grid.z)
  const int t = static_cast<int>(blockIdx.y + gridDim.y * blockIdx.z) * 8 + threadIdx.y;
  if (i >= d / 2 || t >= L) return;
  float c = 0.f, s = 0.f;
  int cur = -1;
  for (int bh = 0; bh < BH; ++bh) {
    const int row = rp.on ? bh / H : 0;
    if (row != cur) {
      angle_cs((rp.on ? rp.p[row] : pos0) + static_cast<float>(t), cc.theta[i], c, s);
      c *= scale;
      s *= scale;
      cur = row;
    }
    const size_t xo = (static_cast<size_t>(bh) * L + ((flip & 1) ? L - 1 - t : t)) * d + 2 * i;
    const size_t yo = (static_cast<size_t>(bh) * L + ((flip & 2) ? L - 1 - t : t)) * d + 2 * i;
    const float a = to_f32(x[xo]);
    const float b = to_f32(x[xo + 1]);
    y[yo] = from_f32<Tout>(a * c - b * s);
    y[yo + 1] = from_f32<Tout>(fmaf(a, s, b * c));
  }
}

// ---------------------------------------------------------------------------
// ΔS_i[k][v] = Σ_j (γ^{r−1−j} k′_j[k]) v_j[v], accumulated in j order from 0.
// Block 16×16 threads, 64 k × 64 v tile, 4×4 outputs per thread.
// grid = (ceil(d_v/64)·F, ceil(d_k/64), ⌈BH·nchunks / F⌉): the (b, h, chunk)
// rows are folded over grid.z and F slices of grid.x (row = blockIdx.z +
// gridDim.z·(blockIdx.x / ceil(d_v/64))); kp = rotated K′ (fp32).
// out: ws[bh][chunk][k][v].
// ---------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(256) chunk_dS_kernel(const float* __restrict__ kp,
                                                       const Tin* __restrict__ v,
                                                       float* __restrict__ ws, CallConsts cc,
                                                       int H, int L, int d_k, int d_v, int chunk,
                                                       int nchunks, int rows) {
  __shared__ float sk[16][64];
  __shared__ float sv[16][64];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * 16 + tx;
  const int ntx = (d_v + 63) / 64;
  const int row = static_cast<int>(blockIdx.z + gridDim.z * (blockIdx.x / ntx));
  if (row >= rows) return;
  const int v0 = static_cast<int>(blockIdx.x % ntx) * 64, k0 = blockIdx.y * 64;
  const int bh = row / nchunks, ci = row % nchunks;
  const int h = bh % H;
  const int start = ci * chunk;
  const int r = min(chunk, L - start);
  const float lg2 = cc.lg2g[h];
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;

  for (int j0 = 0; j0 < r; j0 += 16) {
    for (int e = tid; e < 16 * 64; e += 256) {
      const int jj = e / 64, cc2 = e % 64;
      const int j = j0 + jj;
      float kv = 0.f, vv = 0.f;
      if (j < r) {
        const size_t row = static_cast<size_t>(bh) * L + start + j;
        if (k0 + cc2 < d_k) kv = gpow(lg2, static_cast<float>(r - 1 - j)) * kp[row * d_k + k0 + cc2];
        if (v0 + cc2 < d_v) vv = to_f32(v[row * d_v + v0 + cc2]);
      }
      sk[jj][cc2] = kv;
      sv[jj][cc2] = vv;
    }
    __syncthreads();
    const int jn = min(16, r - j0);
    for (int jj = 0; jj < jn; ++jj) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = sk[jj][ty + 16 * u];
        b[u] = sv[jj][tx + 16 * u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(a[u], b[w], acc[u][w]);
    }
    __syncthreads();
  }
  float* dst = ws + (static_cast<size_t>(bh) * nchunks + ci) * d_k * d_v;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int kk = k0 + ty + 16 * u;
    if (kk >= d_k) continue;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int vv = v0 + tx + 16 * w;
      if (vv < d_v) dst[static_cast<size_t>(kk) * d_v + vv] = acc[u][w];
    }
  }
}

// ---------------------------------------------------------------------------
// Inter-chunk scan over ws[bh][i][k][v] (holding ΔS_i on entry): writes the
// state entering chunk i into slot i and the final state to state_out.
// S_i = fmaf(g, S_{i−1}, ΔS_i) with g = γ^chunk (γ^tail for a ragged last
// chunk), both rounded from double on the host.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) state_scan_kernel(float* __restrict__ ws,
                                                         const float* __restrict__ state_in,
                                                         float* __restrict__ state_out,
                                                         CallConsts cc,
                                                         int H, int d_k, int d_v, int nchunks,
                                                         int BH) {
  const size_t per = static_cast<size_t>(d_k) * d_v;
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= per * BH) return;
  const size_t bh = idx / per, e = idx % per;
  const int h = static_cast<int>(bh % H);
  float S = state_in ? state_in[idx] : 0.f;
  float* p = ws + bh * nchunks * per + e;
  // Sixteen chunks' ΔS are loaded before any of them is combined, so the
  // loads overlap instead of waiting one after another.
  constexpr int PF = 16;
  for (int i0 = 0; i0 < nchunks; i0 += PF) {
    float d[PF];
#pragma unroll
    for (int u = 0; u < PF; ++u)
      if (i0 + u < nchunks) d[u] = p[static_cast<size_t>(i0 + u) * per];
#pragma unroll
    for (int u = 0; u < PF; ++u) {
      const int i = i0 + u;
      if (i < nchunks) {
        p[static_cast<size_t>(i) * per] = S;
        const float g = (i == nchunks - 1) ? cc.gtail[h] : cc.gb[h];
        S = fmaf(g, S, d[u]);
      }
    }
  }
  if (state_out) state_out[idx] = S;
}

// ---------------------------------------------------------------------------
// Per-chunk outputs: o_j = γ^{j+1} q′_j S + Σ_{m≤j} γ^{j−m}(q′_j·k′_m) v_m.
// Block 256 threads = 16 rows × 16 column-threads (4 v each); 64 v per block.
// grid = (ceil(d_v/64), ceil(chunk/16), BH·nchunks).  S = ws slot of the
// chunk (state entering it) or, when ws_states == nullptr, state_in / 0.
// Writes o to out (Tout) or to an fp32 buffer when out_f32 != nullptr.
// ---------------------------------------------------------------------------
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) chunk_out_kernel(
    const float* __restrict__ qp, const float* __restrict__ kp, const Tin* __restrict__ v,
    const float* __restrict__ ws_states, const float* __restrict__ state_in,
    Tout* __restrict__ out, float* __restrict__ out_f32, CallConsts cc, int H, int L, int d_k,
    int d_v, int chunk, int nchunks, int rows) {
  extern __shared__ float smem[];
  float* sq = smem;                 // [16][d_k]
  float* sp = smem + 16 * d_k;      // [16][64] scores
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int ntx = (d_v + 63) / 64;   // rows folded as in chunk_dS_kernel
  const int row = static_cast<int>(blockIdx.z + gridDim.z * (blockIdx.x / ntx));
  if (row >= rows) return;
  const int v0 = static_cast<int>(blockIdx.x % ntx) * 64;
  const int bh = row / nchunks, ci = row % nchunks;
  const int h = bh % H;
  const int start = ci * chunk;
  const int r = min(chunk, L - start);
  const int j0 = blockIdx.y * 16;
  if (j0 >= r) return;
  const float lg2 = cc.lg2g[h];
  const size_t rowbase = static_cast<size_t>(bh) * L + start;

  for (int e = threadIdx.x; e < 16 * d_k; e += 256) {
    const int jj = e / d_k, kk = e % d_k;
    sq[e] = (j0 + jj < r) ? qp[(rowbase + j0 + jj) * d_k + kk] : 0.f;
  }
  __syncthreads();

  const int j = j0 + ty;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  // cross-chunk term q′_j S (ξ applied below)
  const float* S = ws_states ? ws_states + (static_cast<size_t>(bh) * nchunks + ci) * d_k * d_v
                             : (state_in ? state_in + static_cast<size_t>(bh) * d_k * d_v : nullptr);
  if (S) {
    for (int kk = 0; kk < d_k; ++kk) {
      const float qv = sq[ty * d_k + kk];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int vv = v0 + tx + 16 * u;
        if (vv < d_v) o[u] = fmaf(qv, S[static_cast<size_t>(kk) * d_v + vv], o[u]);
      }
    }
    const float xi = gpow(lg2, static_cast<float>(j + 1));
#pragma unroll
    for (int u = 0; u < 4; ++u) o[u] *= xi;
  }
  // intra-chunk term over key tiles of 64
  const int mmax = min(r, j0 + 16);
  for (int m0 = 0; m0 < mmax; m0 += 64) {
    __syncthreads();
    // scores for rows j0..j0+15, keys m0..m0+63: 4 per thread
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int mm = tx + 16 * u;
      const int m = m0 + mm;
      float sc = 0.f;
      if (m < r && m <= j && j < r) {
        const float* kr = kp + (rowbase + m) * d_k;
        const float* qr = sq + ty * d_k;
        float acc = 0.f;
        for (int kk = 0; kk < d_k; ++kk) acc = fmaf(qr[kk], kr[kk], acc);
        sc = acc * gpow(lg2, static_cast<float>(j - m));
      }
      sp[ty * 64 + mm] = sc;
    }
    __syncthreads();
    const int mn = min(64, mmax - m0);
    for (int mm = 0; mm < mn; ++mm) {
      const float pv = sp[ty * 64 + mm];
      const size_t vrow = (rowbase + m0 + mm) * d_v;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int vv = v0 + tx + 16 * u;
        if (vv < d_v) o[u] = fmaf(pv, to_f32(v[vrow + vv]), o[u]);
      }
    }
  }
  if (j >= r) return;
  const size_t orow = (rowbase + j) * d_v;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int vv = v0 + tx + 16 * u;
    if (vv >= d_v) continue;
    if (out_f32) out_f32[orow + vv] = o[u];
    else out[orow + vv] = from_f32<Tout>(o[u]);
  }
}

// ---------------------------------------------------------------------------
// GroupNorm over d_v for each (b, h, t) row: one warp per row.
// («从RoPE到Retention…» §5; one group per head, biased variance.)  y may be
// x itself (same type): every value is read by the lane that writes it, and
// the reductions between the passes order all reads before any write.
// ---------------------------------------------------------------------------
template <typename Tx, typename Tout>
__global__ void __launch_bounds__(256) groupnorm_kernel(const Tx* x, Tout* y,
                                                        const float* __restrict__ w,
                                                        const float* __restrict__ b, int H,
                                                        int L, int d_v, size_t rows, float eps) {
  const size_t row = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int h = static_cast<int>((row / L) % H);
  const Tx* xr = x + row * d_v;
  float s = 0.f;
  for (int c = lane; c < d_v; c += 32) s += to_f32(xr[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mu = s / static_cast<float>(d_v);
  float q = 0.f;
  for (int c = lane; c < d_v; c += 32) {
    const float dlt = to_f32(xr[c]) - mu;
    q = fmaf(dlt, dlt, q);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  const float rstd = rsqrtf(q / static_cast<float>(d_v) + eps);
  Tout* yr = y + row * d_v;
  for (int c = lane; c < d_v; c += 32) {
    float val = (to_f32(xr[c]) - mu) * rstd;
    if (w) val *= w[h * d_v + c];
    if (b) val += b[h * d_v + c];
    yr[c] = from_f32<Tout>(val);
  }
}

// ---------------------------------------------------------------------------
// Decode step («从RoPE到Retention…» §4.2):  S ← γ S + k′ᵀv ;  o = q′ S (new S).
// One block per (b, h); thread t owns VEC consecutive v columns and walks all
// d_k rows of S once (read, update, write, accumulate o).  S is streamed with
// evict-first hints.  Optional GroupNorm over d_v (block reduction).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 ld_stream4(const float* p) {
  float4 r;
  asm volatile("ld.global.cs.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ void st_stream4(float* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

template <typename Tin, typename Tout, int VEC>
__global__ void __launch_bounds__(256) decode_step_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    float* __restrict__ S, Tout* __restrict__ out, CallConsts cc, int H, int d_k, int d_v,
    float pos, int gn_on, float eps, const float* __restrict__ gw,
    const float* __restrict__ gbias) {
  extern __shared__ float sm[];
  float* qs = sm;           // [d_k]
  float* ks = sm + d_k;     // [d_k]
  float* red = sm + 2 * d_k;  // [64]
  const int bh = blockIdx.x;
  const int h = bh % H;
  const int tid = threadIdx.x;
  for (int i = tid; i < d_k / 2; i += blockDim.x) {
    float c, s;
    angle_cs(pos, cc.theta[i], c, s);
    const size_t off = static_cast<size_t>(bh) * d_k + 2 * i;
    const float q0 = to_f32(q[off]), q1 = to_f32(q[off + 1]);
    const float k0 = to_f32(k[off]), k1 = to_f32(k[off + 1]);
    qs[2 * i] = q0 * c - q1 * s;
    qs[2 * i + 1] = fmaf(q0, s, q1 * c);
    ks[2 * i] = cc.kscale * (k0 * c - k1 * s);
    ks[2 * i + 1] = cc.kscale * fmaf(k0, s, k1 * c);
  }
  __syncthreads();
  const float g = cc.gamma[h];
  const int c0 = tid * VEC;
  const bool active = c0 < d_v;
  float vv[VEC], o[VEC];
#pragma unroll
  for (int u = 0; u < VEC; ++u) {
    vv[u] = active ? to_f32(v[static_cast<size_t>(bh) * d_v + c0 + u]) : 0.f;
    o[u] = 0.f;
  }
  float* Sp = S + static_cast<size_t>(bh) * d_k * d_v + c0;
  if (active) {
    if constexpr (VEC == 4) {
      constexpr int U = 8;
      int kk = 0;
      for (; kk + U <= d_k; kk += U) {
        float4 sv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) sv[u] = ld_stream4(Sp + static_cast<size_t>(kk + u) * d_v);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float kv = ks[kk + u], qv = qs[kk + u];
          sv[u].x = fmaf(g, sv[u].x, kv * vv[0]);
          sv[u].y = fmaf(g, sv[u].y, kv * vv[1]);
          sv[u].z = fmaf(g, sv[u].z, kv * vv[2]);
          sv[u].w = fmaf(g, sv[u].w, kv * vv[3]);
          st_stream4(Sp + static_cast<size_t>(kk + u) * d_v, sv[u]);
          o[0] = fmaf(qv, sv[u].x, o[0]);
          o[1] = fmaf(qv, sv[u].y, o[1]);
          o[2] = fmaf(qv, sv[u].z, o[2]);
          o[3] = fmaf(qv, sv[u].w, o[3]);
        }
      }
      for (; kk < d_k; ++kk) {
        float4 s4 = ld_stream4(Sp + static_cast<size_t>(kk) * d_v);
        const float kv = ks[kk], qv = qs[kk];
        s4.x = fmaf(g, s4.x, kv * vv[0]);
        s4.y = fmaf(g, s4.y, kv * vv[1]);
        s4.z = fmaf(g, s4.z, kv * vv[2]);
        s4.w = fmaf(g, s4.w, kv * vv[3]);
        st_stream4(Sp + static_cast<size_t>(kk) * d_v, s4);
        o[0] = fmaf(qv, s4.x, o[0]);
        o[1] = fmaf(qv, s4.y, o[1]);
        o[2] = fmaf(qv, s4.z, o[2]);
        o[3] = fmaf(qv, s4.w, o[3]);
      }
    } else {
      for (int kk = 0; kk < d_k; ++kk) {
        float* p = Sp + static_cast<size_t>(kk) * d_v;
        const float sn = fmaf(g, *p, ks[kk] * vv[0]);
        *p = sn;
        o[0] = fmaf(qs[kk], sn, o[0]);
      }
    }
  }
  if (gn_on) {
    // block mean / variance over the d_v outputs of this (b, h)
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < VEC; ++u) s += active ? o[u] : 0.f;
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if ((tid & 31) == 0) red[tid >> 5] = s;
    __syncthreads();
    float tot = 0.f;
    for (int w2 = 0; w2 < (blockDim.x + 31) / 32; ++w2) tot += red[w2];
    const float mu = tot / static_cast<float>(d_v);
    __syncthreads();
    float q2 = 0.f;
#pragma unroll
    for (int u = 0; u < VEC; ++u) q2 += active ? (o[u] - mu) * (o[u] - mu) : 0.f;
    for (int off = 16; off > 0; off >>= 1) q2 += __shfl_xor_sync(0xffffffffu, q2, off);
    if ((tid & 31) == 0) red[32 + (tid >> 5)] = q2;
    __syncthreads();
    float totq = 0.f;
    for (int w2 = 0; w2 < (blockDim.x + 31) / 32; ++w2) totq += red[32 + w2];
    const float rstd = rsqrtf(totq / static_cast<float>(d_v) + eps);
#pragma unroll
    for (int u = 0; u < VEC; ++u) {
      float val = (o[u] - mu) * rstd;
      if (gw) val *= active ? gw[h * d_v + c0 + u] : 1.f;
      if (gbias) val += active ? gbias[h * d_v + c0 + u] : 0.f;
      o[u] = val;
    }
  }
  if (active) {
#pragma unroll
    for (int u = 0; u < VEC; ++u) out[static_cast<size_t>(bh) * d_v + c0 + u] = from_f32<Tout>(o[u]);
  }
}

// ---------------------------------------------------------------------------
// Row-normalised decay («从RoPE到Retention…» §5, the decay weights normalised
// per row): dividing row N of the decay mask by its sum over the positions
// 0..N it covers, r_N = Σ_{i=0}^{N} γ^i, divides output row N by r_N, so
// the variant is this in-place pass over an output of the plain form:
//   out[bh][t][:] /= r_{pos0+t},  r_N = (1 − γ^{N+1}) / (1 − γ)  (N + 1 at γ = 1)
// r is evaluated as expm1((N+1)·ln γ) / expm1(ln γ), with ln γ from the
// host's double-precision log2 γ, which keeps full relative precision when
// γ is close to 1.  One block of 128 threads per row.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float decay_row_sum(const CallConsts& cc, size_t row, int H, int L,
                                               float pos0) {
  const int t = static_cast<int>(row % L);
  const int h = static_cast<int>((row / L) % H);
  const float lg = cc.lg2g[h] * 0.69314718f;   // ln γ
  const float n1 = pos0 + static_cast<float>(t) + 1.f;
  return lg == 0.f ? n1 : expm1f(n1 * lg) / expm1f(lg);
}

// Any d_v: one block of 128 threads per row, element by element.
template <typename T>
__global__ void __launch_bounds__(128) decay_row_norm_kernel(T* __restrict__ out, CallConsts cc,
                                                             int H, int L, int d_v, float pos0) {
  const size_t row = blockIdx.x;
  const float inv = 1.f / decay_row_sum(cc, row, H, L, pos0);
  T* o = out + row * d_v;
  for (int c = threadIdx.x; c < d_v; c += blockDim.x) o[c] = from_f32<T>(to_f32(o[c]) * inv);
}

// Rows of a whole number of 16-byte vectors (vpr per row): each warp takes 32
// consecutive rows, which are one contiguous run of 32·vpr vectors; lane i
// computes 1/r of row i once, and the run is rewritten in place with 16-byte
// accesses, eight vectors in flight per lane, each multiplied by the 1/r of
// its row (a warp shuffle).  The row of vector e of the run is
// ⌊(e + ½)/vpr⌋ evaluated with one fp32 multiply: e < 32·vpr ≤ 2^14, so the
// product's rounding error (< 2^-9) stays far below the ½/vpr ≥ 2^-10
// distance of the exact quotient to the next integer.  Grid-stride over
// the groups of 32 rows.
template <typename T>
__device__ __forceinline__ uint4 scale_vec(uint4 x, float s);
template <>
__device__ __forceinline__ uint4 scale_vec<float>(uint4 x, float s) {
  return make_uint4(__float_as_uint(__uint_as_float(x.x) * s), __float_as_uint(__uint_as_float(x.y) * s),
                    __float_as_uint(__uint_as_float(x.z) * s), __float_as_uint(__uint_as_float(x.w) * s));
}
template <>
__device__ __forceinline__ uint4 scale_vec<__nv_bfloat16>(uint4 x, float s) {
  auto f = [s](uint32_t w) { return pack_bf16x2(bf16lo_to_f32(w) * s, bf16hi_to_f32(w) * s); };
  return make_uint4(f(x.x), f(x.y), f(x.z), f(x.w));
}

template <typename T>
__global__ void __launch_bounds__(256) decay_row_norm_vec_kernel(uint4* __restrict__ out,
                                                                 CallConsts cc, int H, int L,
                                                                 int vpr, size_t rows, float pos0) {
  constexpr int U = 8;
  const int lane = threadIdx.x & 31;
  const size_t warps = static_cast<size_t>(gridDim.x) * (blockDim.x >> 5);
  for (size_t g = static_cast<size_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       g * 32 < rows; g += warps) {
    const size_t r0 = g * 32;
    const int nr = static_cast<int>(rows - r0 < 32 ? rows - r0 : 32);
    const float inv = lane < nr ? 1.f / decay_row_sum(cc, r0 + lane, H, L, pos0) : 1.f;
    const float rvpr = 1.f / static_cast<float>(vpr);
    uint4* base = out + r0 * vpr;
    const int n = nr * vpr;   // vectors of the run
    for (int e0 = 0; e0 < n; e0 += 32 * U) {
      uint4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = e0 + 32 * u + lane;
        if (e < n) x[u] = __ldcs(base + e);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = e0 + 32 * u + lane;
        const int row = static_cast<int>((static_cast<float>(e < n ? e : 0) + 0.5f) * rvpr);
        const float s = __shfl_sync(0xffffffffu, inv, row);
        if (e < n) __stcs(base + e, scale_vec<T>(x[u], s));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Helpers of the gradient pass (ret_chunkwise_backward).  The gradients are
// three evaluations of the chunkwise form on reordered operands: reading the
// sequence backwards turns the anti-causal sums Σ_{t≥m} of the gradient into
// the causal sums Σ_{m≤t} of the forward form.
// ---------------------------------------------------------------------------
struct HeadScale {
  float s[kMaxHeads];
};

// y[bh, t', c] = x[bh, t, c] converted to Tout, with t' = L−1−t when flip,
// else t.  Grid-stride over the BH·L·d elements (rows contiguous).
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) flip_cvt_kernel(const Tin* __restrict__ x,
                                                       Tout* __restrict__ y, int BH, int L,
                                                       int d, int flip) {
  const size_t n = static_cast<size_t>(BH) * L * d;
  for (size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t row = e / d;
    const int c = static_cast<int>(e - row * d);
    const size_t bh = row / L;
    const int t = static_cast<int>(row - bh * L);
    const size_t dst = (bh * L + (flip ? L - 1 - t : t)) * d + c;
    y[dst] = from_f32<Tout>(to_f32(x[e]));
  }
}

// dst = hs.s[h] · M for BH states src [BH][rows][cols], where M = src or,
// with transpose, srcᵀ ([cols][rows]).  M's rows are cut into pieces of
// prows rows (the last may be shorter); piece p of all BH states comes
// before piece p+1: dst = [piece][BH][rows of the piece][columns of M].
// prows ≥ M's rows gives the plain [BH][M rows][M cols] layout.  src == dst
// only without transpose and pieces (every element is read and written by
// the same thread).  Block (32, 8) per 32×32 tile, grid (⌈cols/32⌉,
// ⌈rows/32⌉, BH); the tile goes through shared memory so that both the
// reads and the (transposed) writes are coalesced.
__global__ void __launch_bounds__(256) state_prep_kernel(const float* src, float* dst, int BH,
                                                         int H, int rows, int cols,
                                                         int transpose, int prows,
                                                         HeadScale hs) {
  __shared__ float tile[32][33];
  const int bh = blockIdx.z;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const float sc = hs.s[bh % H];
  const size_t sb = static_cast<size_t>(bh) * rows * cols;
  const int mrows = transpose ? cols : rows, mcols = transpose ? rows : cols;
  auto dst_index = [&](int mr, int mc) {
    const int piece = mr / prows, rl = mr - piece * prows;
    const int ph = min(prows, mrows - piece * prows);
    return static_cast<size_t>(piece) * prows * mcols * BH +
           (static_cast<size_t>(bh) * ph + rl) * mcols + mc;
  };
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty + 8 * i, c = c0 + tx;
    if (r < rows && c < cols) tile[ty + 8 * i][tx] = src[sb + static_cast<size_t>(r) * cols + c] * sc;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (transpose) {   // M row = source column c0 + ty + 8i, M column = source row r0 + tx
      const int mr = c0 + ty + 8 * i, mc = r0 + tx;
      if (mr < cols && mc < rows) dst[dst_index(mr, mc)] = tile[tx][ty + 8 * i];
    } else {
      const int mr = r0 + ty + 8 * i, mc = c0 + tx;
      if (mr < rows && mc < cols) dst[dst_index(mr, mc)] = tile[ty + 8 * i][tx];
    }
  }
}

// Operands of the tensor-core evaluations in the gradient pass, bf16, all
// derived from one source tensor src [BH][L][d] in one pass:
//   op[bh][t][:] = f(t) · scale · R?((pos0 + t)θ) src[bh][t][:]   (t < L)
//   op[bh][t][:] = 0                                              (L ≤ t < rows_out)
// with the rotation (the prologue's, (cos, sin) of (pos0 + t)·θ_i read from
// the call's table cs [L][d_k/2]) only when rotate.  f(t) is 1 (fold 0),
// ω = γ^{j−(b−1)} (fold 1) or ζ = γ^{b−1−j} (fold 2), j = t mod b, b the
// chunk length: every chunk, the last included, is folded as a whole one
// (rows past L are zero).  Each operand's columns are stored in pieces of
// pw (the last may be narrower), piece-major: [piece][bh][t][columns of the
// piece].  d and pw multiples of 8.
struct OpSpec {
  __nv_bfloat16* dst;
  int rows_out, pw, fold;
  float scale;
};
template <int NS>
struct OpSpecs {
  OpSpec o[NS];
};

// Thread ↔ (row t, 8 columns); threads with t ≥ L zero the padding rows.
// The angles are read once per thread and used for all B·H heads, whose
// loads are issued eight at a time.  NS operands.
template <int NS>
__global__ void __launch_bounds__(256) prep_operand_kernel(
    const __nv_bfloat16* __restrict__ src, OpSpecs<NS> sp, CallConsts cc, const float2* __restrict__ cs,
    int BH, int H, int L, int rows_max, int d, int rotate, int chunk) {
  constexpr int U = 8;
  const int vecs = d / 8;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows_max * vecs) return;
  const int t = idx / vecs, cv = idx - t * vecs;
  auto optr = [&](const OpSpec& o, int bh) {
    const int piece = (8 * cv) / o.pw;
    const int wp = min(o.pw, d - piece * o.pw);
    const size_t at = static_cast<size_t>(piece) * o.pw * o.rows_out * BH +
                      (static_cast<size_t>(bh) * o.rows_out + t) * wp + (8 * cv - piece * o.pw);
    return reinterpret_cast<uint4*>(o.dst + at);
  };
  if (t >= L) {   // padding rows of the operands that have them
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const OpSpec& o = sp.o[i];
      if (t >= o.rows_out) continue;
      for (int bh = 0; bh < BH; ++bh) *optr(o, bh) = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  float c[4] = {1.f, 1.f, 1.f, 1.f}, sn[4] = {0.f, 0.f, 0.f, 0.f};
  if (rotate) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 e = cs[static_cast<size_t>(t) * (d / 2) + 4 * cv + u];
      c[u] = e.x;
      sn[u] = e.y;
    }
  }
  const int j = t % chunk;
  const size_t hstride = static_cast<size_t>(L) * d;
  const __nv_bfloat16* s0 = src + static_cast<size_t>(t) * d + 8 * cv;
  for (int bh0 = 0; bh0 < BH; bh0 += U) {
    uint4 raw[U];
#pragma unroll
    for (int uu = 0; uu < U; ++uu)
      if (bh0 + uu < BH) raw[uu] = __ldcs(reinterpret_cast<const uint4*>(s0 + (bh0 + uu) * hstride));
#pragma unroll
    for (int uu = 0; uu < U; ++uu) {
      const int bh = bh0 + uu;
      if (bh >= BH) break;
      const uint32_t w[4] = {raw[uu].x, raw[uu].y, raw[uu].z, raw[uu].w};
      float r[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float a = bf16lo_to_f32(w[u]), b = bf16hi_to_f32(w[u]);
        r[2 * u] = a * c[u] - b * sn[u];
        r[2 * u + 1] = fmaf(a, sn[u], b * c[u]);
      }
      const float lg = cc.lg2g[bh % H];
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const OpSpec& o = sp.o[i];
        const float ex = o.fold == 1 ? static_cast<float>(j + 1 - chunk) : static_cast<float>(chunk - 1 - j);
        const float f = o.fold ? o.scale * gpow(lg, ex) : o.scale;
        *optr(o, bh) = make_uint4(pack_bf16x2(f * r[0], f * r[1]), pack_bf16x2(f * r[2], f * r[3]),
                                  pack_bf16x2(f * r[4], f * r[5]), pack_bf16x2(f * r[6], f * r[7]));
      }
    }
  }
}

// Gradients from the piece outputs of the evaluations (Tx: fp32, or bf16
// when the gradients are bf16):
//   y[bh][t][:] = scale · R(−(pos0 + t)θ) Σ_{p<np} x[p][bh][t][:]
// with x pieces `pstride` elements apart (summed in fp32) and R(−φ) the
// adjoint (inverse) of the prologue's rotation ((cos, sin) from the call's
// table cs [L][d/2]).  Thread ↔ (row t, 8
// columns), looping over the heads of its group (blockIdx.y).  d a multiple
// of 8.
template <typename Tx>
__device__ __forceinline__ void load8f(const Tx* p, float (&e)[8]) {
  if constexpr (sizeof(Tx) == 2) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e[2 * i] = bf16lo_to_f32(w[i]);
      e[2 * i + 1] = bf16hi_to_f32(w[i]);
    }
  } else {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    e[0] = a.x; e[1] = a.y; e[2] = a.z; e[3] = a.w;
    e[4] = b.x; e[5] = b.y; e[6] = b.z; e[7] = b.w;
  }
}

template <typename Tx, typename Tg>
__global__ void __launch_bounds__(256) grad_out_kernel(const Tx* __restrict__ x,
                                                       size_t pstride, int np,
                                                       Tg* __restrict__ y,
                                                       const float2* __restrict__ cs,
                                                       int BH, int L, int d, float scale) {
  const int vecs = d / 8;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= L * vecs) return;
  const int t = idx / vecs, cv = idx - t * vecs;
  float c[4], sn[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 e = cs[static_cast<size_t>(t) * (d / 2) + 4 * cv + u];
    c[u] = e.x;
    sn[u] = e.y;
  }
  // blockIdx.y: a group of heads (more threads in flight than one loop over all)
  const int hpg = (BH + gridDim.y - 1) / gridDim.y;
  const int bh_end = min(BH, (static_cast<int>(blockIdx.y) + 1) * hpg);
  for (int bh = blockIdx.y * hpg; bh < bh_end; ++bh) {
    const Tx* xr = x + (static_cast<size_t>(bh) * L + t) * d + 8 * cv;
    float e[8];
    load8f(xr, e);
    for (int p = 1; p < np; ++p) {
      float f[8];
      load8f(xr + p * pstride, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) e[i] += f[i];
    }
    float r[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float a = e[2 * u], b = e[2 * u + 1];
      // R(−φ): (a cos φ + b sin φ, b cos φ − a sin φ)
      r[2 * u] = scale * fmaf(a, c[u], b * sn[u]);
      r[2 * u + 1] = scale * fmaf(b, c[u], -a * sn[u]);
    }
    Tg* yr = y + (static_cast<size_t>(bh) * L + t) * d + 8 * cv;
    if constexpr (sizeof(Tg) == 2) {
      *reinterpret_cast<uint4*>(yr) = make_uint4(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]),
                                                 pack_bf16x2(r[4], r[5]), pack_bf16x2(r[6], r[7]));
    } else {
      reinterpret_cast<float4*>(yr)[0] = make_float4(r[0], r[1], r[2], r[3]);
      reinterpret_cast<float4*>(yr)[1] = make_float4(r[4], r[5], r[6], r[7]);
    }
  }
}

// Self-test of the bounded-wait failure path: wait on an mbarrier that no
// one will ever arrive on; the wait must give up and record a timeout.
__global__ void selftest_timeout_kernel(long long budget_cycles) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(1) : "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    for (;;) {
      uint32_t ok;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(a), "r"(0)
          : "memory");
      if (ok) break;
      if (clock64() - t0 > budget_cycles) {
        report_timeout(0xdead0001u);
        break;
      }
    }
  }
}

}  // namespace simt
}  // namespace ret
