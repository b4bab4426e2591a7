// Shared device helpers: status word, bounded waits, bf16 packing, the
// rotation angle of the Θ prologue, per-call constants.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace ret {

constexpr int kMaxHeads = 128;
constexpr int kMaxPairs = 256;   // d_k ≤ 512

// Per-call constants passed by value to every kernel.  Filled on the host
// from the host-side gamma/theta arrays.
// Start position of every batch row when the rows do not share one pos0
// (on = 0: every row starts at the call's pos0).  Positions are exact in fp32.
constexpr int kMaxRowPos = 256;
struct RowPos {
  float p[kMaxRowPos];
  int on;
};

struct CallConsts {
  float theta[kMaxPairs];    // θ_i
  float lg2g[kMaxHeads];     // log2(γ_h), rounded from double
  float gb[kMaxHeads];       // γ_h^chunk, rounded from double (carry factor)
  float gtail[kMaxHeads];    // γ_h^r for the last (possibly shorter) chunk
  float gamma[kMaxHeads];    // γ_h
  float kscale;              // d_k^{-1/2}
};

// ---------------------------------------------------------------------------
// Device status word.  Word 0: error bits (bit 0 = a bounded wait expired);
// word 1: code of the wait that expired; word 2: block index.
// ---------------------------------------------------------------------------
__device__ unsigned int g_ret_status[4];

constexpr unsigned kStatusTimeout = 1u;

__device__ __forceinline__ void report_timeout(unsigned where) {
  if (atomicOr(&g_ret_status[0], kStatusTimeout) == 0) {
    g_ret_status[1] = where;
    g_ret_status[2] = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  }
}

__device__ __forceinline__ bool status_aborted() {
  return *((volatile unsigned int*)&g_ret_status[0]) != 0u;
}

// Wait budget for every spin in the library (cycles of the SM clock).  At the
// B300's 2.03 GHz maximum this is about one second.
constexpr long long kWaitBudgetCycles = 2000000000LL;

// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);   // .x = lo (low 16 bits)
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------
// Rotation angle of the Θ prologue: (cos, sin) of n·θ.
// n < 2^24 is exact in fp32; the product n·θ is split exactly into
// hi + lo (hi = fl(n·θ), lo = fma(n, θ, −hi), |lo| ≤ ulp(hi)/2 ≤ 1 for
// |hi| ≤ 2^24), and sin/cos of the sum follow from the angle-addition
// formulas with CUDA's sincosf of each part.  (A first-order correction for
// lo alone drops lo²/2, which reaches 0.5 near 2^24 rad.)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void angle_cs(float n, float theta, float& c, float& s) {
  const float hi = n * theta;
  const float lo = fmaf(n, theta, -hi);
  float sh, ch, sl, cl;
  sincosf(hi, &sh, &ch);
  sincosf(lo, &sl, &cl);
  s = fmaf(sh, cl, ch * sl);
  c = fmaf(ch, cl, -(sh * sl));
}

// γ^e for a (possibly negative) integer e, from log2 γ: exp2(e·log2 γ).
__device__ __forceinline__ float gpow(float lg2g, float e) { return exp2f(e * lg2g); }

}  // namespace ret
