// libretention.so — C ABI (include/retention.h): argument validation, path
// selection, workspace layout and kernel launches.  One translation unit so
// the device status word and the kernels share a module.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "retention.h"
#include "common.cuh"
#include "tc_primitives.cuh"
#include "kernels_simt.cuh"
#include "kernel_tc_chunk.cuh"
#include "kernel_tc_parallel.cuh"
#include "kernel_tc_pair.cuh"
#include "kernel_tc_gemm.cuh"
#include "kernels_grad.cuh"
#include "kernel_tc_walk.cuh"

using namespace ret;

namespace {

int g_force_path = 0;

// Profiling hook state (see ret_profile_begin).
struct ProfileHook {
  cudaEvent_t* ev = nullptr;
  int cap = 0;
  int used = 0;              // kernels recorded
  const char* names[64] = {};
} g_prof;

// Brackets one kernel launch with the hook's events when it is armed.
// NVTX range around an entry point, for timeline tools (header-only NVTX:
// without an attached tool each push / pop is a no-op call).
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

struct Mark {
  cudaStream_t st;
  bool on;
  Mark(const char* name, cudaStream_t s) : st(s), on(false) {
    if (g_prof.ev && 2 * g_prof.used + 1 < g_prof.cap && g_prof.used < 64) {
      g_prof.names[g_prof.used] = name;
      cudaEventRecord(g_prof.ev[2 * g_prof.used], st);
      on = true;
    }
  }
  ~Mark() {
    if (on) {
      cudaEventRecord(g_prof.ev[2 * g_prof.used + 1], st);
      ++g_prof.used;
    }
  }
};

constexpr int64_t kMaxPos = int64_t(1) << 24;

// Calls whose rows all start at the call's pos0.
RowPos no_rowpos() {
  RowPos r;
  std::memset(&r, 0, sizeof(r));
  return r;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------------------
// Per-call constants from the host arrays γ[H], θ[d_k/2]
// ---------------------------------------------------------------------------
ret_status make_consts(CallConsts& cc, const float* gamma, const float* theta, int H, int d_k,
                       int chunk, int L) {
  std::memset(&cc, 0, sizeof(cc));
  if (!gamma || !theta) return RET_EINVAL;
  for (int i = 0; i < d_k / 2; ++i) {
    if (!std::isfinite(theta[i])) return RET_EINVAL;
    cc.theta[i] = theta[i];
  }
  const int tail = (chunk > 0 && L > 0) ? (L - ((L - 1) / chunk) * chunk) : 0;
  for (int h = 0; h < H; ++h) {
    const double g = gamma[h];
    if (!(g > 0.0) || !(g <= 1.0)) return RET_EINVAL;
    const double lg = std::log2(g);
    cc.gamma[h] = gamma[h];
    cc.lg2g[h] = static_cast<float>(lg);
    cc.gb[h] = static_cast<float>(std::pow(g, static_cast<double>(chunk > 0 ? chunk : 1)));
    cc.gtail[h] = static_cast<float>(std::pow(g, static_cast<double>(tail > 0 ? tail : 1)));
  }
  cc.kscale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k)));
  return RET_OK;
}

ret_status check_common(const void* q, const void* k, const void* v, ret_dtype in_dt, int B,
                        int H, int L, int d_k, int d_v, int64_t pos0, const float* s_in,
                        const float* s_out, const void* out, ret_dtype out_dt, const ret_gn* gn) {
  if (in_dt != RET_F32 && in_dt != RET_BF16) return RET_EINVAL;
  if (out_dt != RET_F32 && out_dt != RET_BF16) return RET_EINVAL;
  if (!q || !k || !v || !out) return RET_EINVAL;
  if (!al16(q) || !al16(k) || !al16(v) || !al16(out)) return RET_EINVAL;
  if ((s_in && !al16(s_in)) || (s_out && !al16(s_out))) return RET_EINVAL;
  if (B < 1 || H < 1 || H > kMaxHeads || L < 1) return RET_EINVAL;
  if (d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) || d_v < 1 || d_v > 1024) return RET_EINVAL;
  if (pos0 < 0 || pos0 + L > kMaxPos) return RET_EINVAL;
  if (static_cast<int64_t>(B) * H * L >= (int64_t(1) << 31)) return RET_EINVAL;
  if (gn && gn->enabled) {
    if (!(gn->eps > 0.f) || !std::isfinite(gn->eps)) return RET_EINVAL;
    if ((gn->weight && !al16(gn->weight)) || (gn->bias && !al16(gn->bias))) return RET_EINVAL;
  }
  return RET_OK;
}

bool gn_on(const ret_gn* gn) { return gn && gn->enabled; }

ret_status cuda_status(cudaError_t e) { return e == cudaSuccess ? RET_OK : RET_ECUDA; }

ret_status last_launch() { return cuda_status(cudaGetLastError()); }

// ---------------------------------------------------------------------------
// TMA descriptors (driver entry point fetched through the runtime)
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qres{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qres) == cudaSuccess &&
        qres == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box 64 × 128, 128-B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
              uint32_t box_rows = 128) {
  if (!get_encode()) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [n][rows][cols] bf16 viewed in 3-D with boxes of 64 columns × box_rows rows
// of one matrix: rows past `rows` read as zeros (never the next matrix's).
bool make_map3(CUtensorMap* m, const void* base, uint64_t n, uint64_t rows, uint64_t cols,
               uint32_t box_rows = 128) {
  if (!get_encode()) return false;
  cuuint64_t dims[3] = {cols, rows, n};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Path choice
// ---------------------------------------------------------------------------
bool tc_gamma_ok(const float* gamma, int H, int chunk) {
  if (!gamma) return true;
  for (int h = 0; h < H; ++h) {
    const double g = gamma[h];
    if (!(g > 0.0) || !(g <= 1.0)) return false;
    // every factor γ^{±(b−1)} of the rewritten form stays within 2^±60
    if (-(chunk - 1) * std::log2(g) > 60.0) return false;
  }
  return true;
}

// The tensor-core chunk kernels: tiles of 128 d_v columns (d_v a multiple
// of 128, or one tile of which the first 64 columns are live) and chunks of
// 128 tokens.  A requested chunk of 64 runs on the same 128-token tiles: the
// chunkwise form's value does not depend on the chunk length (b = 1 gives the
// recurrent form, b = L the parallel one), so only the rounding differs.
bool tc_chunk_ok(ret_dtype in_dt, const float* gamma, int H, int L, int d_k, int d_v,
                 int chunk) {
  if (g_force_path == RET_PATH_SIMT) return false;
  if (in_dt != RET_BF16) return false;
  if (!(d_k == 64 || d_k == 128 || d_k == 256)) return false;
  if ((d_v % tcc::VT != 0 && d_v != 64) || (chunk != tcc::CH && chunk != tcc::CH / 2) || L < 1)
    return false;
  return tc_gamma_ok(gamma, H, tcc::CH);
}

int tc_tiles(int d_v) { return (d_v + tcc::VT - 1) / tcc::VT; }

// CTA pairs (cta_group::2) for the chunk kernels: the two d_v tiles of a
// pair share one head, so d_v must hold an even number of whole tiles.
bool tc_pair_ok(int d_k, int d_v) {
  return g_force_path != RET_PATH_TC_SINGLE && (d_k == 128 || d_k == 256) && d_v % tcc::VT == 0 &&
         (d_v / tcc::VT) % 2 == 0;
}

// Grid rows of the tensor-core launches: B·H (carry layout) or B·H·L/128
// (one chunk per row) must fit gridDim.y.
constexpr size_t kMaxGridRows = 65535;

// Grids whose row count may exceed gridDim.y / gridDim.z (65535).  fold_z:
// the SIMT chunk kernels, rows over grid.z and F slices of grid.x.
// fold_rows: the tensor-core chunk kernels, rows over grid.y and grid.z
// (ChunkArgs::grid_rows set when folded).
dim3 fold_z(unsigned x, unsigned y, size_t rows) {
  const size_t gz = std::min<size_t>(rows, kMaxGridRows);
  const size_t f = (rows + gz - 1) / gz;
  return dim3(static_cast<unsigned>(x * f), y, static_cast<unsigned>(gz));
}

// rotate_kernel: groups of 8 rows over grid.y and grid.z (it drops rows ≥ L).
dim3 fold_y(unsigned x, size_t rows) {
  const size_t gz = (rows + kMaxGridRows - 1) / kMaxGridRows;
  return dim3(x, static_cast<unsigned>((rows + gz - 1) / gz), static_cast<unsigned>(gz));
}

dim3 fold_rows(unsigned x, size_t rows, int* grid_rows) {
  if (rows <= kMaxGridRows) {
    *grid_rows = 0;
    return dim3(x, static_cast<unsigned>(rows));
  }
  const size_t gz = (rows + kMaxGridRows - 1) / kMaxGridRows;
  const size_t gy = (rows + gz - 1) / gz;
  *grid_rows = static_cast<int>(rows);
  return dim3(x, static_cast<unsigned>(gy), static_cast<unsigned>(gz));
}

struct Plan {
  int path = 0;
  size_t bytes = 0;
  // workspace offsets
  size_t off_q = 0, off_k = 0, off_states = 0;
  size_t off_tail = 0;   // staging of a short last chunk's outputs (tensor-core path)
  // Ring mode (carried layout on CTA pairs): off_q / off_k hold the ring of
  // `ring` chunk slots for ring_heads heads; off_flags its counters; off_cs
  // the angle table [L][d_k/2] (cos, sin).
  int ring = 0, ring_heads = 0;
  size_t off_flags = 0, off_cs = 0;
  // ret_chunkwise on the tensor cores in the chunk-parallel layout (a grid
  // of B·H·tiles CTAs too small to keep the SMs busy for the carried one).
  bool scan = false;
};

// The carried layout runs B·H·tiles CTAs that each walk every chunk, one
// chunk time per chunk; the chunk-parallel layout runs two passes of one-chunk
// CTAs (each CTA's life, set-up and pipeline fill included, about three chunk
// times) plus the scan and two more launches (about eight chunk times).  So
// with fewer CTAs than half the SMs, the chunk-parallel layout is chosen when
// 6·⌈B·H·tiles·chunks / 148⌉ + 8 < chunks (measured on eight shapes from 4 to
// 32 carried CTAs and 8 to 128 chunks: it picks the faster layout on all of
// them, within 6% where the two are close).  Both give the same bits.
constexpr size_t kCarryMinCtas = 74;
bool prefer_scan(size_t BH, int d_v, int nch) {
  const size_t ctas = BH * tc_tiles(d_v);
  if (g_force_path != 0 || ctas >= kCarryMinCtas) return false;
  const size_t waves = (ctas * nch + 147) / 148;
  return 6 * waves + 8 < static_cast<size_t>(nch);
}

// Compact-workspace mode of the carried layout on CTA pairs: the Θ prologue
// runs inside the chunk launch (producer CTAs on the SMs the consumer pairs
// leave over, writing an L2-resident ring of chunk slots) instead of as a
// front pass over the whole sequence.  Chunk slots per head in the ring, and
// the most consumer CTAs one ring launch plans for (148 SMs, about a seventh
// of them left to the producers; the launch re-checks co-residency with the
// occupancy query).
constexpr int kRing = 4;
constexpr int kRingConsumers = 128;
constexpr int kRingMaxProducers = 40;

bool ring_mode_ok(int d_k, int d_v) { return tc_pair_ok(d_k, d_v); }


// compact: the compact-workspace mode where it applies (carried layout on
// CTA pairs), else the same plan as without it.
Plan plan_chunkwise(ret_dtype in_dt, const float* gamma, int B, int H, int L, int d_k, int d_v,
                    int chunk, bool gn, bool scan = false, bool compact = false) {
  Plan p;
  const size_t BH = static_cast<size_t>(B) * H;
  const bool tc = tc_chunk_ok(in_dt, gamma, H, L, d_k, d_v, chunk);
  const int nch = (L + (tc ? tcc::CH : chunk) - 1) / (tc ? tcc::CH : chunk);
  size_t off = 0;
  if (tc) {
    p.path = RET_PATH_TC;
    if (compact && !scan && ring_mode_ok(d_k, d_v)) {
      // producer ring: kRing chunk slots of Q″ and K̂′ per head of one launch,
      // the launch's counters and the call's angle table
      const int ntiles = tc_tiles(d_v);
      p.ring = kRing;
      p.ring_heads = static_cast<int>(std::min<size_t>(BH, std::max(1, kRingConsumers / ntiles)));
      const size_t slots = static_cast<size_t>(p.ring_heads) * kRing * tcc::CH * d_k * 2;
      p.off_flags = off; off += 256;
      p.off_q = off; off += up256(slots);
      p.off_k = off; off += up256(slots);
      p.off_cs = off; off += up256(static_cast<size_t>(L) * (d_k / 2) * 8);
    } else {
      // rotated Q′ / K̂′, each sequence padded with zero rows to whole chunks
      const size_t Lp = static_cast<size_t>(nch) * tcc::CH;
      p.off_q = off; off += up256(BH * Lp * d_k * 2);
      p.off_k = off; off += up256(BH * Lp * d_k * 2);
    }
    if (!scan && !p.ring && prefer_scan(BH, d_v, nch)) p.scan = true;
    if (scan || p.scan) { p.off_states = off; off += up256(BH * nch * static_cast<size_t>(d_k) * d_v * 4); }
    if (L % tcc::CH != 0) { p.off_tail = off; off += up256(BH * tcc::CH * static_cast<size_t>(d_v) * 4); }
  } else {
    p.path = RET_PATH_SIMT;
    p.off_q = off; off += up256(BH * L * d_k * 4);
    p.off_k = off; off += up256(BH * L * d_k * 4);
    p.off_states = off; off += up256(BH * nch * static_cast<size_t>(d_k) * d_v * 4);
  }
  p.bytes = off;
  return p;
}

Plan plan_parallel(ret_dtype in_dt, const float* gamma, int B, int H, int L, int d_k, int d_v,
                   bool gn, bool want_state) {
  Plan p;
  const size_t BH = static_cast<size_t>(B) * H;
  size_t off = 0;
  if (tc_chunk_ok(in_dt, gamma, H, L, d_k, d_v, tcc::CH) && d_v % tcc::VT == 0 && L % tcc::CH == 0 &&
      BH <= kMaxGridRows && static_cast<size_t>(L / tcc::CH) <= kMaxGridRows) {   // parallel_tc grid (·, BH, blocks)
    // rotated Q′ / K̂′ in bf16; per-block ΔS states when state_out is wanted
    p.path = RET_PATH_TC;
    p.off_q = off; off += up256(BH * L * d_k * 2);
    p.off_k = off; off += up256(BH * L * d_k * 2);
    if (want_state) {
      p.off_states = off;
      off += up256(BH * (L / tcc::CH) * static_cast<size_t>(d_k) * d_v * 4);
    }
    p.bytes = off;
    return p;
  }
  p.path = RET_PATH_SIMT;
  p.off_q = off; off += up256(BH * L * d_k * 4);
  p.off_k = off; off += up256(BH * L * d_k * 4);
  if (want_state) { p.off_states = off; off += up256(BH * static_cast<size_t>(d_k) * d_v * 4); }
  p.bytes = off;
  return p;
}

// GroupNorm over the rows of x into y (y may be x when Tx = Ty): rows in
// registers when d_v is a multiple of 8 (eight 256-thread blocks per SM's
// worth of warps at most, grid-stride over the row groups), else one warp
// per row.
template <typename Tx, typename Ty, int NV>
void launch_gn_forward_reg(const Tx* x, Ty* y, const ret_gn* gn, int H, int L, int d_v, size_t rows,
                           cudaStream_t st) {
  const size_t blocks = std::min<size_t>((rows + 7) / 8, static_cast<size_t>(148) * 8);
  grad::gn_forward_reg_kernel<Tx, Ty, NV><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      x, y, gn->weight, gn->bias, H, L, d_v, rows, gn->eps);
}

template <typename Tx, typename Ty>
void launch_groupnorm(const Tx* x, Ty* y, const ret_gn* gn, int H, int L, int d_v, size_t rows,
                      cudaStream_t st) {
  Mark m("groupnorm", st);
  if (d_v % 8 != 0) {
    simt::groupnorm_kernel<Tx, Ty><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
        x, y, gn->weight, gn->bias, H, L, d_v, rows, gn->eps);
  } else if (d_v <= 256) {
    launch_gn_forward_reg<Tx, Ty, 8>(x, y, gn, H, L, d_v, rows, st);
  } else if (d_v <= 512) {
    launch_gn_forward_reg<Tx, Ty, 16>(x, y, gn, H, L, d_v, rows, st);
  } else {
    launch_gn_forward_reg<Tx, Ty, 32>(x, y, gn, H, L, d_v, rows, st);
  }
}

template <typename T> T* wsp(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// ---------------------------------------------------------------------------
// fp32 path: rotation into fp32 workspace, per-chunk ΔS, scan, outputs
// ---------------------------------------------------------------------------
template <typename Tin, typename Tout>
ret_status run_simt_chunked(const Tin* q, const Tin* k, const Tin* v, const CallConsts& cc,
                            int B, int H, int L, int d_k, int d_v, int64_t pos0, int chunk,
                            const float* s_in, float* s_out, Tout* out, const ret_gn* gn,
                            void* ws, const Plan& p, bool need_states, cudaStream_t st,
                            const RowPos& rp) {
  const int BH = B * H;
  const int nch = (L + chunk - 1) / chunk;
  float* qp = wsp<float>(ws, p.off_q);
  float* kp = wsp<float>(ws, p.off_k);
  {
    const dim3 grid = fold_y((d_k / 2 + 31) / 32, (static_cast<size_t>(L) + 7) / 8);
    {
      Mark m("rotate_q_f32", st);
      simt::rotate_kernel<Tin, float><<<grid, dim3(32, 8), 0, st>>>(q, qp, cc, BH, H, L, d_k,
                                                                    static_cast<float>(pos0), 1.f, rp, 0);
    }
    {
      Mark m("rotate_k_f32", st);
      simt::rotate_kernel<Tin, float><<<grid, dim3(32, 8), 0, st>>>(k, kp, cc, BH, H, L, d_k,
                                                                    static_cast<float>(pos0), cc.kscale, rp, 0);
    }
  }
  float* states = need_states ? wsp<float>(ws, p.off_states) : nullptr;
  if (states) {
    const dim3 g1 = fold_z((d_v + 63) / 64, (d_k + 63) / 64, static_cast<size_t>(BH) * nch);
    {
      Mark m("chunk_dS_f32", st);
      simt::chunk_dS_kernel<Tin><<<g1, dim3(16, 16), 0, st>>>(kp, v, states, cc, H, L, d_k, d_v,
                                                              chunk, nch, BH * nch);
    }
    const size_t n = static_cast<size_t>(BH) * d_k * d_v;
    Mark m("state_scan", st);
    simt::state_scan_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
        states, s_in, s_out, cc, H, d_k, d_v, nch, BH);
  }
  {
    const dim3 g2 = fold_z((d_v + 63) / 64, (chunk + 15) / 16, static_cast<size_t>(BH) * nch);
    const size_t smem = (16 * static_cast<size_t>(d_k) + 16 * 64) * sizeof(float);
    // ws_states == nullptr means "use state_in for the single chunk" (parallel form)
    const float* wst = (nch > 1 || states) ? states : nullptr;
    Mark m("chunk_out_f32", st);
    simt::chunk_out_kernel<Tin, Tout><<<g2, 256, smem, st>>>(qp, kp, v, wst, s_in, out, nullptr, cc,
                                                             H, L, d_k, d_v, chunk, nch, BH * nch);
  }
  if (gn_on(gn))   // in place over out
    launch_groupnorm<Tout, Tout>(out, out, gn, H, L, d_v, static_cast<size_t>(BH) * L, st);
  return last_launch();
}

// ---------------------------------------------------------------------------
// Ring mode: the Θ prologue fused into the CTA-pair launch
// ---------------------------------------------------------------------------
// Largest number of clusters of two pair-kernel CTAs that can be resident at
// once on the current device (0 if the query fails), cached per device.
constexpr int kMaxDev = 64;

template <int DK>
int pair_max_clusters() {
  static std::mutex mu;
  static int cache[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] > 0) return cache[dev];
  const uint32_t smem = tcq::Cfg<DK>::SMEM_BYTES;
  if (cudaFuncSetAttribute(tcq::pair_tc_kernel<DK, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 128);
  cfg.blockDim = dim3(tcc::NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tcq::pair_tc_kernel<DK, true>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cache[dev] = n;
  return n;
}

// [n][rows][cols] bf16 read in boxes of one row of `cols` × `box_n` matrices
// (no swizzle): the raw q / k rows of the ring producers.
bool make_map_rows(CUtensorMap* m, const void* base, uint64_t n, uint64_t rows, uint64_t cols,
                   uint32_t box_n) {
  if (!get_encode()) return false;
  cuuint64_t dims[3] = {cols, rows, n};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(cols), 1, box_n};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Carried layout on CTA pairs with the Θ prologue inside the launch.  The
// heads run in groups sized so that every CTA of a launch is resident at
// once: per group, producer CTAs (the SMs the consumer pairs leave over, at
// most kRingMaxProducers) rotate raw q, k into the ring and the consumer
// pairs read it from there (kernel_tc_pair.cuh, ring_producer).  The ring's
// counters are cleared before each group's launch.  Q″ and K̂′ are the front
// pass's values bit for bit, so results equal the front-pass path's.
template <int DK, typename Tout>
ret_status run_tc_ring(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
                       const CallConsts& cc, int B, int H, int L, int d_v, int64_t pos0,
                       const float* s_in, float* s_out, Tout* out, const ret_gn* gn, void* ws,
                       const Plan& p, cudaStream_t st, const RowPos& rp) {
  using CfgP = tcq::Cfg<DK>;
  const int BH = B * H;
  const int nch = (L + tcc::CH - 1) / tcc::CH;
  const int Lp = nch * tcc::CH;
  const int ntiles = d_v / tcc::VT;
  const int ncl = pair_max_clusters<DK>();
  const int per_row = 2 * ncl / ntiles;          // grid rows that fit at once
  const int G = std::min(p.ring_heads, per_row - 1);
  if (G < 1) return RET_EUNSUPPORTED;
  uint32_t* flags = wsp<uint32_t>(ws, p.off_flags);
  auto* rq = wsp<__nv_bfloat16>(ws, p.off_q);
  auto* rk = wsp<__nv_bfloat16>(ws, p.off_k);
  auto* cs = wsp<float2>(ws, p.off_cs);
  if (!rp.on) {
    const size_t n = static_cast<size_t>(L) * (DK / 2);
    Mark m("angle_table", st);
    tcc::angle_table_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
        cs, cc, L, DK / 2, static_cast<float>(pos0));
    if (cudaGetLastError() != cudaSuccess) return RET_ECUDA;
  }
  const uint64_t ring_rows = static_cast<uint64_t>(p.ring_heads) * kRing * tcc::CH;
  CUtensorMap mqh, mkh, mk, mv, mrq, mrk;
  if (!make_map(&mqh, rq, ring_rows, DK, 64) || !make_map(&mkh, rk, ring_rows, DK, 64) ||
      !make_map(&mk, rk, ring_rows, DK) ||
      !make_map3(&mv, v, static_cast<uint64_t>(BH), static_cast<uint64_t>(L), d_v))
    return RET_ECUDA;
  tcc::ChunkArgs a;
  a.state_in = s_in;
  a.state_out = s_out;
  a.out = static_cast<void*>(out);
  a.out_f32 = sizeof(Tout) == 4 ? 1 : 0;
  a.H = H;
  a.d_v = d_v;
  a.nchunks = nch;
  a.seq_len = L;
  a.seq_lp = Lp;
  a.seq_chunks = nch;
  a.tail_out = (L % tcc::CH != 0) ? wsp<void>(ws, p.off_tail) : nullptr;
  a.seq_div = 1;
  a.raw_ds = 0;
  a.ring = kRing;
  a.ring_flags = flags;
  a.ring_q = rq;
  a.ring_k = rk;
  a.ring_cs = cs;
  const uint32_t smem = CfgP::SMEM_BYTES;
  if (cudaFuncSetAttribute(tcq::pair_tc_kernel<DK, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return RET_ECUDA;
  for (int bh0 = 0; bh0 < BH; bh0 += G) {
    const int Gl = std::min(G, BH - bh0);
    const int prod_rows = std::min(per_row - Gl, std::max(1, kRingMaxProducers / ntiles));
    const uint32_t stride = (2u * Gl * DK * 2 + DK * 4 + 1023u) & ~1023u;
    const int nbuf = static_cast<int>(std::min<uint32_t>(4, (CfgP::USED - 256) / stride));
    if (nbuf < 2) return RET_EUNSUPPORTED;
    if (!make_map_rows(&mrq, q, static_cast<uint64_t>(BH), static_cast<uint64_t>(L), DK, Gl) ||
        !make_map_rows(&mrk, k, static_cast<uint64_t>(BH), static_cast<uint64_t>(L), DK, Gl))
      return RET_ECUDA;
    a.ring_prod_rows = prod_rows;
    a.ring_heads = Gl;
    a.ring_bh0 = bh0;
    a.ring_npairs = Gl * ntiles / 2;
    a.ring_nbuf = nbuf;
    if (cudaMemsetAsync(flags, 0, 2 * kRing * sizeof(uint32_t), st) != cudaSuccess) return RET_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ntiles, prod_rows + Gl);
    cfg.blockDim = dim3(tcc::NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    Mark m("chunk_tc_ring", st);
    if (cudaLaunchKernelEx(&cfg, tcq::pair_tc_kernel<DK, true>, mqh, mkh, mk, mv, mrq, mrk, a, cc, rp) !=
        cudaSuccess)
      return RET_ECUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return RET_ECUDA;
  if (a.tail_out) {   // the short last chunk's valid rows, from the staging tile
    const int T = L - (nch - 1) * tcc::CH;
    const int row_vecs = d_v * (a.out_f32 ? 4 : 2) / 16;
    const size_t n = static_cast<size_t>(BH) * T * row_vecs;
    Mark m("tail_copy", st);
    tcc::tail_copy_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
        static_cast<const uint4*>(a.tail_out), static_cast<uint4*>(a.out), BH, T, L, (nch - 1) * tcc::CH,
        row_vecs);
    if (cudaGetLastError() != cudaSuccess) return RET_ECUDA;
  }
  if (gn_on(gn))   // in place over out
    launch_groupnorm<Tout, Tout>(out, out, gn, H, L, d_v, static_cast<size_t>(BH) * L, st);
  return last_launch();
}

// scan = false: one CTA walks all chunks of its (b, h), carrying the state.
// scan = true: chunk-parallel layout — every chunk's ΔS from zero (one CTA
// per chunk), the fp32 scan over chunks, then every chunk's outputs from its
// entering state.  Both run the same kernel code, so state and outputs agree
// bit for bit.
// parallel = true (ret_parallel): the parallel-form kernel computes the
// outputs, and state_out (if wanted) comes from the ΔS + scan steps.
template <typename Tout>
ret_status run_tc_chunk(const __nv_bfloat16* q, const __nv_bfloat16* k, const __nv_bfloat16* v,
                        const CallConsts& cc, int B, int H, int L, int d_k, int d_v,
                        int64_t pos0, const float* s_in, float* s_out, Tout* out,
                        const ret_gn* gn, void* ws, const Plan& p, cudaStream_t st,
                        const RowPos& rp, bool scan = false, bool parallel = false,
                        bool prerot = false) {
  if (p.ring && !scan && !parallel)
    return d_k == 256 ? run_tc_ring<256, Tout>(q, k, v, cc, B, H, L, d_v, pos0, s_in, s_out, out, gn, ws, p, st, rp)
                      : run_tc_ring<128, Tout>(q, k, v, cc, B, H, L, d_v, pos0, s_in, s_out, out, gn, ws, p, st, rp);
  const int BH = B * H;
  __nv_bfloat16* qr = wsp<__nv_bfloat16>(ws, p.off_q);
  __nv_bfloat16* kr = wsp<__nv_bfloat16>(ws, p.off_k);
  const int nch = (L + tcc::CH - 1) / tcc::CH;
  const int Lp = nch * tcc::CH;   // rows per sequence in the rotated workspace
  if (!prerot) {   // (prerot: the workspace already holds Q″ and K̂′)
    const size_t n = static_cast<size_t>(Lp) * (d_k / 8);
    Mark m("rotate_qk_bf16", st);
    const unsigned bx = static_cast<unsigned>((n + 255) / 256);
    const unsigned by = static_cast<unsigned>(std::max<size_t>(
        1, std::min<size_t>((static_cast<size_t>(BH) + 7) / 8, (2 * 148 + bx - 1) / bx)));
    tcc::rotate_qk_kernel<<<dim3(bx, by), 256, 0, st>>>(
        q, k, qr, kr, cc, BH, H, L, Lp, d_k, static_cast<float>(pos0), tcc::CH, parallel ? 0 : 1, rp);
  }
  // Q′ / K̂′: the padded workspace, flat; V: [B·H][L][d_v] in 3-D for the
  // chunk kernels (a short last chunk reads zeros past L), flat for the
  // parallel form (L a multiple of 128 there).
  CUtensorMap mq, mk, mv, mv2;
  const uint64_t rows = static_cast<uint64_t>(BH) * Lp;
  if (!make_map(&mq, qr, rows, d_k) || !make_map(&mk, kr, rows, d_k) ||
      !make_map3(&mv, v, static_cast<uint64_t>(BH), static_cast<uint64_t>(L), d_v) ||
      (parallel && !make_map(&mv2, v, static_cast<uint64_t>(BH) * L, d_v)))
    return RET_ECUDA;
  const bool pair = tc_pair_ok(d_k, d_v);
  CUtensorMap mqh, mkh;   // 64-row boxes of Q′ / K̂′ for the pair kernel
  if (pair && (!make_map(&mqh, qr, rows, d_k, 64) || !make_map(&mkh, kr, rows, d_k, 64)))
    return RET_ECUDA;
  tcc::ChunkArgs a;
  a.state_in = s_in;
  a.state_out = s_out;
  a.out = static_cast<void*>(out);
  a.out_f32 = sizeof(Tout) == 4 ? 1 : 0;
  a.H = H;
  a.d_v = d_v;
  a.nchunks = nch;
  a.seq_len = L;
  a.seq_lp = Lp;
  a.seq_chunks = nch;
  a.tail_out = (L % tcc::CH != 0 && a.out) ? wsp<void>(ws, p.off_tail) : nullptr;
  a.seq_div = 1;
  a.raw_ds = 0;
  auto launch = [&](auto kern, uint32_t smem, const tcc::ChunkArgs& args0, int rows,
                    const char* name) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    tcc::ChunkArgs args = args0;
    const dim3 grid = fold_rows(tc_tiles(d_v), static_cast<size_t>(rows), &args.grid_rows);
    Mark m(name, st);
    kern<<<grid, tcc::NTHREADS, smem, st>>>(mq, mk, mv, args, cc);
    return cudaGetLastError();
  };
  // Pair kernel: clusters of two CTAs along the d_v tiles.
  auto launch_pair = [&](auto kern, uint32_t smem, const tcc::ChunkArgs& args0, int rows,
                         const char* name) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    tcc::ChunkArgs args = args0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = fold_rows(d_v / tcc::VT, static_cast<size_t>(rows), &args.grid_rows);
    cfg.blockDim = dim3(tcc::NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    Mark m(name, st);
    e = cudaLaunchKernelEx(&cfg, kern, mqh, mkh, mk, mv, mk, mk, args, cc, rp);
    return e != cudaSuccess ? e : cudaGetLastError();
  };
  // Grids of more than 65535 rows take the instantiations that fold them.
  auto run = [&](const tcc::ChunkArgs& args, int rows, const char* name) -> cudaError_t {
    constexpr int F = tcc::kModeFold;
    const bool fold = static_cast<size_t>(rows) > kMaxGridRows;
    if (pair && d_k == 256)
      return fold ? launch_pair(tcq::pair_tc_kernel<256, false, F>, tcq::Cfg<256>::SMEM_BYTES, args, rows, name)
                  : launch_pair(tcq::pair_tc_kernel<256, false>, tcq::Cfg<256>::SMEM_BYTES, args, rows, name);
    if (pair)
      return fold ? launch_pair(tcq::pair_tc_kernel<128, false, F>, tcq::Cfg<128>::SMEM_BYTES, args, rows, name)
                  : launch_pair(tcq::pair_tc_kernel<128, false>, tcq::Cfg<128>::SMEM_BYTES, args, rows, name);
    if (d_k == 256)
      return fold ? launch(tcc::chunk_tc_kernel<256, F>, tcc::Cfg<256>::SMEM_BYTES, args, rows, name)
                  : launch(tcc::chunk_tc_kernel<256>, tcc::Cfg<256>::SMEM_BYTES, args, rows, name);
    if (d_k == 128)
      return fold ? launch(tcc::chunk_tc_kernel<128, F>, tcc::Cfg<128>::SMEM_BYTES, args, rows, name)
                  : launch(tcc::chunk_tc_kernel<128>, tcc::Cfg<128>::SMEM_BYTES, args, rows, name);
    return fold ? launch(tcc::chunk_tc_kernel<64, F>, tcc::Cfg<64>::SMEM_BYTES, args, rows, name)
                : launch(tcc::chunk_tc_kernel<64>, tcc::Cfg<64>::SMEM_BYTES, args, rows, name);
  };
  cudaError_t e = cudaSuccess;
  if (parallel) {
    tcp::ParArgs pa;
    pa.state_in = s_in;
    pa.out = a.out;
    pa.out_f32 = a.out_f32;
    pa.H = H;
    pa.L = L;
    pa.d_v = d_v;
    auto plaunch = [&](auto kern, uint32_t smem) -> cudaError_t {
      cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem));
      if (e2 != cudaSuccess) return e2;
      Mark m("parallel_tc", st);
      kern<<<dim3(d_v / tcp::VT, BH, nch), tcp::NTHREADS, smem, st>>>(mq, mk, mv2, pa, cc);
      return cudaGetLastError();
    };
    if (d_k == 256) e = plaunch(tcp::parallel_tc_kernel<256>, tcp::Cfg<256>::SMEM_BYTES);
    else if (d_k == 128) e = plaunch(tcp::parallel_tc_kernel<128>, tcp::Cfg<128>::SMEM_BYTES);
    else e = plaunch(tcp::parallel_tc_kernel<64>, tcp::Cfg<64>::SMEM_BYTES);
    if (e == cudaSuccess && s_out) {   // closed-form final state: ΔS per block, then the scan
      float* states = wsp<float>(ws, p.off_states);
      tcc::ChunkArgs d = a;
      d.nchunks = 1;
      d.seq_div = nch;
      d.raw_ds = 1;
      d.state_in = nullptr;
      d.state_out = states;
      d.out = nullptr;
      d.tail_out = nullptr;
      e = run(d, BH * nch, "chunk_tc_dS");
      if (e == cudaSuccess) {
        const size_t n = static_cast<size_t>(BH) * d_k * d_v;
        Mark m("state_scan", st);
        simt::state_scan_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
            states, s_in, s_out, cc, H, d_k, d_v, nch, BH);
        e = cudaGetLastError();
      }
    }
  } else if (!scan) {
    e = run(a, BH, "chunk_tc");
  } else {
    // The [BH, L, d] tensors viewed as [BH·nch, 128, d]: one chunk per row.
    float* states = wsp<float>(ws, p.off_states);
    tcc::ChunkArgs d = a;
    d.nchunks = 1;
    d.seq_div = nch;
    d.raw_ds = 1;
    d.state_in = nullptr;
    d.state_out = states;   // ΔS of every chunk
    d.out = nullptr;
    d.tail_out = nullptr;
    e = run(d, BH * nch, "chunk_tc_dS");
    if (e == cudaSuccess) {
      const size_t n = static_cast<size_t>(BH) * d_k * d_v;
      Mark m("state_scan", st);
      simt::state_scan_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
          states, s_in, s_out, cc, H, d_k, d_v, nch, BH);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) {
      tcc::ChunkArgs o = a;
      o.nchunks = 1;
      o.seq_div = nch;
      o.state_in = states;    // state entering every chunk
      o.state_out = nullptr;
      e = run(o, BH * nch, "chunk_tc_out");
    }
  }
  if (e != cudaSuccess) return RET_ECUDA;
  if (a.tail_out && !parallel) {   // the short last chunk's valid rows, from the staging tile
    const int T = L - (nch - 1) * tcc::CH;
    const int row_vecs = d_v * (a.out_f32 ? 4 : 2) / 16;
    const size_t n = static_cast<size_t>(BH) * T * row_vecs;
    Mark m("tail_copy", st);
    tcc::tail_copy_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
        static_cast<const uint4*>(a.tail_out), static_cast<uint4*>(a.out), BH, T, L, (nch - 1) * tcc::CH,
        row_vecs);
    if (cudaGetLastError() != cudaSuccess) return RET_ECUDA;
  }
  if (gn_on(gn))   // in place over out
    launch_groupnorm<Tout, Tout>(out, out, gn, H, L, d_v, static_cast<size_t>(BH) * L, st);
  return last_launch();
}

template <typename Tin>
ret_status dispatch_simt_out(const void* q, const void* k, const void* v, const CallConsts& cc,
                             int B, int H, int L, int d_k, int d_v, int64_t pos0, int chunk,
                             const float* s_in, float* s_out, void* out, ret_dtype out_dt,
                             const ret_gn* gn, void* ws, const Plan& p, bool need_states,
                             cudaStream_t st, const RowPos& rp) {
  const Tin* qq = static_cast<const Tin*>(q);
  const Tin* kk = static_cast<const Tin*>(k);
  const Tin* vv = static_cast<const Tin*>(v);
  if (out_dt == RET_F32)
    return run_simt_chunked<Tin, float>(qq, kk, vv, cc, B, H, L, d_k, d_v, pos0, chunk, s_in,
                                        s_out, static_cast<float*>(out), gn, ws, p, need_states, st,
                                        rp);
  return run_simt_chunked<Tin, __nv_bfloat16>(qq, kk, vv, cc, B, H, L, d_k, d_v, pos0, chunk,
                                               s_in, s_out, static_cast<__nv_bfloat16*>(out), gn,
                                               ws, p, need_states, st, rp);
}

// ---------------------------------------------------------------------------
// Gradient pass (fp32 kernels)
// ---------------------------------------------------------------------------
// Workspace: rotated Q′ (reversed), K′ (in order and reversed), dO and V in
// fp32 (in order — only for bf16 inputs, fp32 inputs are read in place — and
// reversed), one fp32 output of the forward-form evaluations, the per-chunk
// states of those evaluations, and one prepared d×d state.
struct BwdPlan {
  size_t off_qpf = 0, off_kp = 0, off_kpf = 0, off_do = 0, off_dof = 0, off_v = 0, off_vf = 0;
  size_t off_fout = 0, off_states = 0, off_sprep = 0, bytes = 0;
};

BwdPlan plan_backward(ret_dtype in_dt, int B, int H, int L, int d_k, int d_v, int chunk) {
  BwdPlan p;
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t nch = (static_cast<size_t>(L) + chunk - 1) / chunk;
  const size_t rk = up256(BH * L * d_k * 4), rv = up256(BH * L * static_cast<size_t>(d_v) * 4);
  size_t off = 0;
  p.off_qpf = off; off += rk;
  p.off_kp = off; off += rk;
  p.off_kpf = off; off += rk;
  if (in_dt == RET_BF16) {
    p.off_do = off; off += rv;
    p.off_v = off; off += rv;
  }
  p.off_dof = off; off += rv;
  p.off_vf = off; off += rv;
  p.off_fout = off; off += up256(BH * L * static_cast<size_t>(d_k > d_v ? d_k : d_v) * 4);
  p.off_states = off; off += up256(BH * nch * static_cast<size_t>(d_k) * d_v * 4);
  p.off_sprep = off; off += up256(BH * static_cast<size_t>(d_k) * d_v * 4);
  p.bytes = off;
  return p;
}

unsigned stride_grid(size_t n) {
  const size_t b = (n + 255) / 256;
  return static_cast<unsigned>(b < 148 * 16 ? (b > 0 ? b : 1) : 148 * 16);
}

// One evaluation of the chunkwise form on fp32 operands that are already
// rotated and scaled (no Θ step): out = o(qp, kp, v; s_in), s_out optional.
// qp, kp: [BH, L, dk]; v, out: [BH, L, dv]; states: [BH, nch, dk, dv].
ret_status run_simt_core(const float* qp, const float* kp, const float* v, const CallConsts& cc,
                         int BH, int H, int L, int dk, int dv, int chunk, const float* s_in,
                         float* s_out, float* out, float* states, cudaStream_t st) {
  const int nch = (L + chunk - 1) / chunk;
  const bool need = nch > 1 || s_out;
  if (need) {
    const dim3 g1 = fold_z((dv + 63) / 64, (dk + 63) / 64, static_cast<size_t>(BH) * nch);
    {
      Mark m("bwd_chunk_dS", st);
      simt::chunk_dS_kernel<float><<<g1, dim3(16, 16), 0, st>>>(kp, v, states, cc, H, L, dk, dv,
                                                                chunk, nch, BH * nch);
    }
    const size_t n = static_cast<size_t>(BH) * dk * dv;
    Mark m("bwd_state_scan", st);
    simt::state_scan_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
        states, s_in, s_out, cc, H, dk, dv, nch, BH);
  }
  const dim3 g2 = fold_z((dv + 63) / 64, (chunk + 15) / 16, static_cast<size_t>(BH) * nch);
  const size_t smem = (16 * static_cast<size_t>(dk) + 16 * 64) * sizeof(float);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(simt::chunk_out_kernel<float, float>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return RET_ECUDA;
  Mark m("bwd_chunk_out", st);
  simt::chunk_out_kernel<float, float><<<g2, 256, smem, st>>>(qp, kp, v, need ? states : nullptr,
                                                              s_in, out, nullptr, cc, H, L, dk,
                                                              dv, chunk, nch, BH * nch);
  return last_launch();
}

// Gradients of o and S_out with respect to q, k, v, S_in, per head with the
// decay mask A, ξ_t = γ^{t+1}, w_m = γ^{L−1−m} and G = (dO Vᵀ) ⊙ A (the
// chain rule on the parallel form of «从RoPE到Retention…» §4.1 with the state
// terms):
//   dQ′ = G K′ + ξ ⊙ (dO S_inᵀ)            dV = (Q′K′ᵀ ⊙ A)ᵀ dO + (w ⊙ K′) dS_out
//   dK′ = Gᵀ Q′ + (w ⊙ V) dS_outᵀ           dS_in = (ξ ⊙ Q′)ᵀ dO + γ^L dS_out
// Each is one evaluation F(a, b, c; S) of the chunkwise form (o_t =
// Σ_{m≤t} γ^{t−m}(a_t·b_m) c_m + γ^{t+1} a_t S, S_out = γ^L S + Σ γ^{L−1−m}
// b_mᵀ c_m): dQ′ = F(dO, V, K′; S_inᵀ); over the reversed sequence (↓),
// dV↓ = F(K′↓, Q′↓, dO↓; dS_out/γ) with dS_in = γ · its S_out, and
// dK′↓ = F(V↓, dO↓, Q′↓; dS_outᵀ/γ).  Then dq = R(−nθ) dQ′ and
// dk = d_k^{-1/2} R(−nθ) dK′ (R is orthogonal).
template <typename Tin, typename Tg>
ret_status run_backward(const Tin* q, const Tin* k, const Tin* v, const Tin* d_o,
                        const CallConsts& cc, int B, int H, int L, int d_k, int d_v,
                        int64_t pos0, int chunk, const float* s_in, const float* dso, Tg* dq,
                        Tg* dk, Tg* dv, float* dsi, void* ws, const BwdPlan& p,
                        cudaStream_t st) {
  const int BH = B * H;
  float* qpf = wsp<float>(ws, p.off_qpf);
  float* kp = wsp<float>(ws, p.off_kp);
  float* kpf = wsp<float>(ws, p.off_kpf);
  float* dof = wsp<float>(ws, p.off_dof);
  float* vf = wsp<float>(ws, p.off_vf);
  float* fout = wsp<float>(ws, p.off_fout);
  float* states = wsp<float>(ws, p.off_states);
  float* sprep = wsp<float>(ws, p.off_sprep);
  const RowPos rp = no_rowpos();
  const float p0 = static_cast<float>(pos0);
  const dim3 rg = fold_y((d_k / 2 + 31) / 32, (static_cast<size_t>(L) + 7) / 8);
  const size_t nk = static_cast<size_t>(BH) * L * d_k, nv = static_cast<size_t>(BH) * L * d_v;
  const dim3 sgrid((d_v + 31) / 32, (d_k + 31) / 32, BH);   // state_prep_kernel tiles
  {
    Mark m("bwd_rotate", st);
    simt::rotate_kernel<Tin, float><<<rg, dim3(32, 8), 0, st>>>(q, qpf, cc, BH, H, L, d_k, p0,
                                                                1.f, rp, 2);
  }
  {
    Mark m("bwd_rotate", st);
    simt::rotate_kernel<Tin, float><<<rg, dim3(32, 8), 0, st>>>(k, kp, cc, BH, H, L, d_k, p0,
                                                                cc.kscale, rp, 0);
  }
  {
    Mark m("bwd_flip", st);
    simt::flip_cvt_kernel<float, float><<<stride_grid(nk), 256, 0, st>>>(kp, kpf, BH, L, d_k, 1);
  }
  const float* do32;
  const float* v32;
  if constexpr (std::is_same<Tin, float>::value) {
    do32 = d_o;
    v32 = v;
  } else {   // bf16 inputs: fp32 copies in order
    float* a = wsp<float>(ws, p.off_do);
    float* b = wsp<float>(ws, p.off_v);
    {
      Mark m("bwd_flip", st);
      simt::flip_cvt_kernel<Tin, float><<<stride_grid(nv), 256, 0, st>>>(d_o, a, BH, L, d_v, 0);
    }
    {
      Mark m("bwd_flip", st);
      simt::flip_cvt_kernel<Tin, float><<<stride_grid(nv), 256, 0, st>>>(v, b, BH, L, d_v, 0);
    }
    do32 = a;
    v32 = b;
  }
  {
    Mark m("bwd_flip", st);
    simt::flip_cvt_kernel<Tin, float><<<stride_grid(nv), 256, 0, st>>>(d_o, dof, BH, L, d_v, 1);
  }
  {
    Mark m("bwd_flip", st);
    simt::flip_cvt_kernel<Tin, float><<<stride_grid(nv), 256, 0, st>>>(v, vf, BH, L, d_v, 1);
  }
  simt::HeadScale one, ginv, gam;
  for (int h = 0; h < kMaxHeads; ++h) {
    one.s[h] = 1.f;
    ginv.s[h] = h < H ? static_cast<float>(1.0 / static_cast<double>(cc.gamma[h])) : 1.f;
    gam.s[h] = h < H ? cc.gamma[h] : 1.f;
  }
  CallConsts ca = cc;   // R(−nθ): the same angles with θ negated
  for (int i = 0; i < kMaxPairs; ++i) ca.theta[i] = -cc.theta[i];
  ret_status s;
  // dQ′ = F(dO, V, K′; S_inᵀ), then dq = R(−nθ) dQ′
  const float* x = nullptr;
  if (s_in) {
    Mark m("bwd_state_prep", st);
    simt::state_prep_kernel<<<sgrid, dim3(32, 8), 0, st>>>(s_in, sprep, BH, H, d_k, d_v, 1, d_v, one);
    x = sprep;
  }
  if ((s = run_simt_core(do32, v32, kp, cc, BH, H, L, d_v, d_k, chunk, x, nullptr, fout, states,
                         st)) != RET_OK)
    return s;
  {
    Mark m("bwd_rotate", st);
    simt::rotate_kernel<float, Tg><<<rg, dim3(32, 8), 0, st>>>(fout, dq, ca, BH, H, L, d_k, p0,
                                                               1.f, rp, 0);
  }
  // dK′↓ = F(V↓, dO↓, Q′↓; dS_outᵀ/γ), then dk = d_k^{-1/2} R(−nθ) dK′
  x = nullptr;
  if (dso) {
    Mark m("bwd_state_prep", st);
    simt::state_prep_kernel<<<sgrid, dim3(32, 8), 0, st>>>(dso, sprep, BH, H, d_k, d_v, 1, d_v, ginv);
    x = sprep;
  }
  if ((s = run_simt_core(vf, dof, qpf, cc, BH, H, L, d_v, d_k, chunk, x, nullptr, fout, states,
                         st)) != RET_OK)
    return s;
  {
    Mark m("bwd_rotate", st);
    simt::rotate_kernel<float, Tg><<<rg, dim3(32, 8), 0, st>>>(fout, dk, ca, BH, H, L, d_k, p0,
                                                               cc.kscale, rp, 1);
  }
  // dV↓ = F(K′↓, Q′↓, dO↓; dS_out/γ) and dS_in = γ · S_out of that evaluation.
  // dS_out is read (into sprep) before dS_in is written, so the two may alias.
  x = nullptr;
  if (dso) {
    Mark m("bwd_state_prep", st);
    simt::state_prep_kernel<<<sgrid, dim3(32, 8), 0, st>>>(dso, sprep, BH, H, d_k, d_v, 0, d_k, ginv);
    x = sprep;
  }
  if ((s = run_simt_core(kpf, qpf, dof, cc, BH, H, L, d_k, d_v, chunk, x, dsi, fout, states,
                         st)) != RET_OK)
    return s;
  {
    Mark m("bwd_flip", st);
    simt::flip_cvt_kernel<float, Tg><<<stride_grid(nv), 256, 0, st>>>(fout, dv, BH, L, d_v, 1);
  }
  if (dsi) {
    Mark m("bwd_state_prep", st);
    simt::state_prep_kernel<<<sgrid, dim3(32, 8), 0, st>>>(dsi, dsi, BH, H, d_k, d_v, 0, d_k, gam);
  }
  return last_launch();
}

// ---------------------------------------------------------------------------
// Gradient pass on the tensor cores (bf16 inputs): the same three
// evaluations, run by the chunk kernels on operands that prep_operand_kernel
// lays out as the front pass lays out Q″ and K̂′, with one difference: every
// chunk, the last included, is folded as a whole chunk of 128 rows (ω_j =
// γ^{j−127}, ζ_j = γ^{127−j}, j the row within the chunk; rows past L are
// zero).  The sequence is then evaluated as if it had Lp rows, and:
//  * the forward evaluation (dQ′) gives the same outputs when the last chunk
//    carries with γ^128 too (only its final state, which is not used, is
//    scaled);
//  * the anti-causal evaluations (dK′, dV) run on the chunk kernels' reverse
//    mode (last chunk first, keys m ≥ j) with the query operand folded by ζ
//    and the key operand by ω: their scores are γ^{m−j} a_j·b_m, and the
//    kernel's state is γ^{−127} times the state of the anti-causal recursion
//    R ← γ^128 R + Σ_m γ^m b_m c_mᵀ started at row Lp.  So the dK′ evaluation
//    reads the dQ′ evaluation's two folded operands with their roles
//    exchanged (ζ·V as queries, ω·dO as keys), the dV evaluation reads K̂′ and
//    Q″ as queries and keys and dO itself as values, and both start from
//    γ^{−127}·γ^{r−128}·dS_out/γ (r the last chunk's length: dS_out/γ is the
//    state at row L, γ^{r−128} moves it to row Lp) and dS_in = γ^128 · the
//    final state.  The evaluations whose scores contract over d_v run as a
//    sum of pieces of at most 256 columns (the scores are linear in the
//    contracted columns, and so is the cross term once the state is cut by
//    the same rows).  When every piece is 256 wide, the pieces run in one
//    launch as extra grid rows (piece p of (b, h) is row p·B·H + b·H + h),
//    which keeps enough CTAs in flight when d_k = 256 gives only two d_v
//    tiles per row; those rows read one copy of the value operand.
// ---------------------------------------------------------------------------
constexpr int kBwdPiece = 256;

int bwd_pieces(int d_v) { return (d_v + kBwdPiece - 1) / kBwdPiece; }

bool tc_backward_ok(ret_dtype in_dt, const float* gamma, int H, int d_k, int d_v, int chunk,
                    int B) {
  if (g_force_path == RET_PATH_SIMT || in_dt != RET_BF16 || chunk != tcc::CH) return false;
  if (!(d_k == 128 || d_k == 256) || d_v % tcc::VT != 0) return false;
  if (!tc_gamma_ok(gamma, H, chunk)) return false;
  // the reverse evaluations' states carry factors up to γ^{−255}: keep them
  // within 2^100
  for (int h = 0; gamma && h < H; ++h)
    if (-(2 * chunk - 1) * std::log2(static_cast<double>(gamma[h])) > 100.0) return false;
  return true;
}

struct TcBwdPlan {
  // operands: ω·dO and ζ·V (dQ′ and, roles exchanged, dK′; 256-column
  // pieces), K′ (dQ′'s values), Q′ (dK′'s values), K̂′ and Q″ (dV's queries
  // and keys)
  size_t off_dof = 0, off_vf = 0, off_kr = 0, off_qr = 0, off_kf = 0, off_qf = 0;
  size_t off_x = 0, off_sprep = 0, off_cs = 0, off_tail = 0, bytes = 0;
  int pieces = 0;
  bool as_rows = false;   // all pieces in one launch
};

TcBwdPlan plan_tc_backward(int B, int H, int L, int d_k, int d_v) {
  TcBwdPlan p;
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t Lp = static_cast<size_t>((L + tcc::CH - 1) / tcc::CH) * tcc::CH;
  p.pieces = bwd_pieces(d_v);
  p.as_rows = d_v % kBwdPiece == 0;
  const size_t xw = std::max(static_cast<size_t>(p.pieces) * d_k, static_cast<size_t>(d_v));
  const size_t av = up256(BH * Lp * d_v * 2), ak = up256(BH * Lp * d_k * 2);
  const size_t ck = up256(BH * L * d_k * 2);
  size_t off = 0;
  p.off_dof = off; off += av;
  p.off_vf = off; off += av;
  p.off_kr = off; off += ck;
  p.off_qr = off; off += ck;
  p.off_kf = off; off += ak;
  p.off_qf = off; off += ak;
  p.off_x = off; off += up256(BH * L * static_cast<size_t>(p.pieces) * d_k * 4);   // fp32, per piece
  p.off_sprep = off; off += up256(BH * static_cast<size_t>(d_k) * d_v * 4);
  p.off_cs = off; off += up256(static_cast<size_t>(L) * (d_k / 2) * sizeof(float2));   // angle table
  if (L % tcc::CH != 0) { p.off_tail = off; off += up256(BH * tcc::CH * xw * 4); }
  p.bytes = off;
  return p;
}

// out ([rows][L][dvF], fp32 or bf16) = the chunkwise form over `rows`
// sequences with Q″ = a and K̂′ = b (bf16 [rows][Lp][dkF]), V = c (bf16
// [rows mod v_seqs][L][dvF], v_seqs 0: [rows]); s_in / s_out per row
// [dkF][dvF], the starting state read as γ^s_in_exp · s_in and the final
// one written as γ^s_out_exp · S.  Head of row r: r mod H.  rev: the
// reverse mode (anti-causal).
ret_status run_tc_eval(const __nv_bfloat16* a, const __nv_bfloat16* b, int dkF,
                       const __nv_bfloat16* c, int dvF, int v_seqs, const float* s_in,
                       int s_in_exp, float* s_out, int s_out_exp, void* out, int out_f32,
                       void* tail, const CallConsts& cc, int rows, int H, int L, bool rev,
                       cudaStream_t st) {
  const int nch = (L + tcc::CH - 1) / tcc::CH;
  const int Lp = nch * tcc::CH;
  const uint64_t qrows = static_cast<uint64_t>(rows) * Lp;
  const bool pair = tc_pair_ok(dkF, dvF);
  const uint64_t vrows = static_cast<uint64_t>(v_seqs ? v_seqs : rows);
  CUtensorMap mq, mk, mv, mqh, mkh;
  if (!make_map(&mq, a, qrows, dkF) || !make_map(&mk, b, qrows, dkF) ||
      !make_map3(&mv, c, vrows, static_cast<uint64_t>(L), dvF))
    return RET_ECUDA;
  if (pair && (!make_map(&mqh, a, qrows, dkF, 64) || !make_map(&mkh, b, qrows, dkF, 64)))
    return RET_ECUDA;
  tcc::ChunkArgs g;
  g.state_in = s_in;
  g.state_out = s_out;
  g.out = out;
  g.out_f32 = out_f32;
  g.H = H;
  g.d_v = dvF;
  g.nchunks = nch;
  g.seq_len = L;
  g.seq_lp = Lp;
  g.seq_chunks = nch;
  g.tail_out = (L % tcc::CH != 0) ? tail : nullptr;
  g.seq_div = 1;
  g.raw_ds = 0;
  g.v_seqs = v_seqs;
  g.s_in_exp = s_in_exp;
  g.s_out_exp = s_out_exp;
  auto launch_pair = [&](auto kern, uint32_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = fold_rows(dvF / tcc::VT, static_cast<size_t>(rows), &g.grid_rows);
    cfg.blockDim = dim3(tcc::NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    Mark m("bwd_chunk_tc", st);
    e = cudaLaunchKernelEx(&cfg, kern, mqh, mkh, mk, mv, mk, mk, g, cc, no_rowpos());
    return e != cudaSuccess ? e : cudaGetLastError();
  };
  auto launch = [&](auto kern, uint32_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid = fold_rows(tc_tiles(dvF), static_cast<size_t>(rows), &g.grid_rows);
    Mark m("bwd_chunk_tc", st);
    kern<<<grid, tcc::NTHREADS, smem, st>>>(mq, mk, mv, g, cc);
    return cudaGetLastError();
  };
  cudaError_t e;
  // the gradient pass's instantiations (they also fold grids of more than
  // 65535 rows)
  constexpr int FW = tcc::kModeBwd | tcc::kModeFold, RV = FW | tcc::kModeRev;
  if (pair && dkF == 256)
    e = rev ? launch_pair(tcq::pair_tc_kernel<256, false, RV>, tcq::Cfg<256>::SMEM_BYTES)
            : launch_pair(tcq::pair_tc_kernel<256, false, FW>, tcq::Cfg<256>::SMEM_BYTES);
  else if (pair)
    e = rev ? launch_pair(tcq::pair_tc_kernel<128, false, RV>, tcq::Cfg<128>::SMEM_BYTES)
            : launch_pair(tcq::pair_tc_kernel<128, false, FW>, tcq::Cfg<128>::SMEM_BYTES);
  else if (dkF == 256)
    e = rev ? launch(tcc::chunk_tc_kernel<256, RV>, tcc::Cfg<256>::SMEM_BYTES)
            : launch(tcc::chunk_tc_kernel<256, FW>, tcc::Cfg<256>::SMEM_BYTES);
  else
    e = rev ? launch(tcc::chunk_tc_kernel<128, RV>, tcc::Cfg<128>::SMEM_BYTES)
            : launch(tcc::chunk_tc_kernel<128, FW>, tcc::Cfg<128>::SMEM_BYTES);
  if (e != cudaSuccess) return RET_ECUDA;
  if (g.tail_out) {
    const int T = L - (nch - 1) * tcc::CH;
    const int row_vecs = dvF * (out_f32 ? 4 : 2) / 16;
    const size_t n = static_cast<size_t>(rows) * T * row_vecs;
    Mark m("bwd_tail_copy", st);
    tcc::tail_copy_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
        static_cast<const uint4*>(g.tail_out), static_cast<uint4*>(out), rows, T, L,
        (nch - 1) * tcc::CH, row_vecs);
  }
  return last_launch();
}

template <typename Tg>
ret_status run_tc_backward(const __nv_bfloat16* q, const __nv_bfloat16* k,
                           const __nv_bfloat16* v, const __nv_bfloat16* d_o, const CallConsts& cc0,
                           int B, int H, int L, int d_k, int d_v, int64_t pos0, const float* s_in,
                           const float* dso, Tg* dq, Tg* dk, Tg* dv, float* dsi, void* ws,
                           const TcBwdPlan& p, cudaStream_t st) {
  const int BH = B * H;
  const int nch = (L + tcc::CH - 1) / tcc::CH;
  const int Lp = nch * tcc::CH;
  const int r = L - (nch - 1) * tcc::CH;   // rows of the last chunk
  CallConsts cc = cc0;                     // every chunk carries as a whole one
  for (int h = 0; h < H; ++h) cc.gtail[h] = cc.gb[h];
  auto op = [&](size_t off) { return wsp<__nv_bfloat16>(ws, off); };
  // dQ′, dK′ pieces in the gradients' type (the workspace is sized for fp32)
  Tg* X = wsp<Tg>(ws, p.off_x);
  constexpr int x_f32 = sizeof(Tg) == 4;
  float* sprep = wsp<float>(ws, p.off_sprep);
  void* tail = p.off_tail ? wsp<void>(ws, p.off_tail) : nullptr;
  const size_t nk = static_cast<size_t>(BH) * L * d_k;
  // (cos, sin) of (pos0 + t)·θ_i once for the call: the operand pass and the
  // gradient outputs read it
  float2* cs = wsp<float2>(ws, p.off_cs);
  {
    Mark m("bwd_angles", st);
    const size_t n = static_cast<size_t>(L) * (d_k / 2);
    tcc::angle_table_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
        cs, cc, L, d_k / 2, static_cast<float>(pos0));
  }
  // All operands, one pass per source tensor.
  auto prep = [&](const __nv_bfloat16* src, int d, int rotate, const auto& sp) {
    const int n = Lp * (d / 8);
    Mark m("bwd_prep", st);
    constexpr int NS = sizeof(sp.o) / sizeof(sp.o[0]);
    simt::prep_operand_kernel<NS><<<(n + 255) / 256, 256, 0, st>>>(src, sp, cc, cs, BH, H, L, Lp, d,
                                                                   rotate, tcc::CH);
  };
  //                                   dst            rows pw         fold scale
  prep(d_o, d_v, 0, simt::OpSpecs<1>{{{op(p.off_dof), Lp, kBwdPiece, 1, 1.f}}});
  prep(v, d_v, 0, simt::OpSpecs<1>{{{op(p.off_vf), Lp, kBwdPiece, 2, 1.f}}});
  prep(k, d_k, 1, simt::OpSpecs<2>{{{op(p.off_kr), L, d_k, 0, cc.kscale},
                                    {op(p.off_kf), Lp, d_k, 2, cc.kscale}}});
  prep(q, d_k, 1, simt::OpSpecs<2>{{{op(p.off_qr), L, d_k, 0, 1.f},
                                    {op(p.off_qf), Lp, d_k, 1, 1.f}}});
  // gradient = scale · R(−nθ) Σ pieces of X
  auto grad_out = [&](Tg* y, float scale) {
    Mark m("bwd_grad_out", st);
    const unsigned groups = static_cast<unsigned>(std::min(BH, 4));
    simt::grad_out_kernel<Tg, Tg><<<dim3((L * (d_k / 8) + 255) / 256, groups), 256, 0, st>>>(
        X, nk, p.pieces, y, cs, BH, L, d_k, scale);
  };
  // dst = scale_h · (S or Sᵀ), cut into pieces of prows rows
  auto state_prep = [&](const float* src, float* dst, int transpose, int prows,
                        const simt::HeadScale& hs) {
    Mark m("bwd_state_prep", st);
    simt::state_prep_kernel<<<dim3((d_v + 31) / 32, (d_k + 31) / 32, BH), dim3(32, 8), 0, st>>>(
        src, dst, BH, H, d_k, d_v, transpose, prows, hs);
  };
  const int start_exp = r - 2 * tcc::CH;   // γ^{−127}·γ^{r−128}/γ
  simt::HeadScale one, start;
  for (int h = 0; h < kMaxHeads; ++h) {
    const double g = h < H ? static_cast<double>(cc.gamma[h]) : 1.0;
    one.s[h] = 1.f;
    start.s[h] = static_cast<float>(std::pow(g, start_exp));
  }
  ret_status s;
  // The evaluations that contract over d_v: a, b piece-major, c the values,
  // s_pieces the pieces of the starting state; piece outputs land nk apart
  // in X.
  auto pieces = [&](const __nv_bfloat16* a, const __nv_bfloat16* b, const __nv_bfloat16* c,
                    const float* s_pieces, bool rev) -> ret_status {
    if (p.as_rows)
      return run_tc_eval(a, b, kBwdPiece, c, d_k, BH, s_pieces, 0, nullptr, 0, X, x_f32, tail, cc,
                         p.pieces * BH, H, L, rev, st);
    for (int pc = 0; pc < p.pieces; ++pc) {
      const int c0 = pc * kBwdPiece;
      const int w = std::min(kBwdPiece, d_v - c0);
      const size_t ob = static_cast<size_t>(c0) * Lp * BH;   // piece base in a, b
      const float* sp = s_pieces ? s_pieces + static_cast<size_t>(c0) * d_k * BH : nullptr;
      ret_status rs = run_tc_eval(a + ob, b + ob, w, c, d_k, 0, sp, 0, nullptr, 0,
                                  X + static_cast<size_t>(pc) * nk, x_f32, tail, cc, BH, H, L, rev, st);
      if (rs != RET_OK) return rs;
    }
    return RET_OK;
  };
  // dQ′ = F(ω·dO, ζ·V, K′; S_inᵀ), then dq = R(−nθ) dQ′
  if (s_in) state_prep(s_in, sprep, 1, kBwdPiece, one);
  if ((s = pieces(op(p.off_dof), op(p.off_vf), op(p.off_kr), s_in ? sprep : nullptr, false)) !=
      RET_OK)
    return s;
  grad_out(dq, 1.f);
  // dK′ = reverse F(ζ·V, ω·dO, Q′; start·dS_outᵀ), then dk = d_k^{-1/2} R(−nθ) dK′
  if (dso) state_prep(dso, sprep, 1, kBwdPiece, start);
  if ((s = pieces(op(p.off_vf), op(p.off_dof), op(p.off_qr), dso ? sprep : nullptr, true)) !=
      RET_OK)
    return s;
  grad_out(dk, cc.kscale);
  // dV = reverse F(K̂′, Q″, dO; γ^start_exp·dS_out), written in place, and
  // dS_in = γ^128 · its final state (each drain thread reads its elements of
  // dS_out before it writes the same elements of dS_in, so the two may alias)
  if ((s = run_tc_eval(op(p.off_kf), op(p.off_qf), d_k, d_o, d_v, 0, dso, start_exp, dsi, tcc::CH,
                       dv, x_f32, tail, cc, BH, H, L, true, st)) != RET_OK)
    return s;
  return last_launch();
}

// ---------------------------------------------------------------------------
// MSR block: projections (tcgen05 GEMMs with fused epilogues), the chunkwise
// core on the projected operands, GroupNorm with the swish gate, the output
// projection.
// ---------------------------------------------------------------------------
struct BlockPlan {
  Plan core;            // the chunkwise core (front-pass layout; Q″ / K̂′ come from the GEMMs)
  size_t off_cs = 0, off_v = 0, off_o = 0, off_g = 0, off_a = 0, bytes = 0;
  bool ok = false;
};

BlockPlan plan_block(const float* gamma, int B, int L, int D, int H, int d_k, int d_v, int D_out) {
  BlockPlan bp;
  bp.core = plan_chunkwise(RET_BF16, gamma, B, H, L, d_k, d_v, tcc::CH, false);
  bp.ok = bp.core.path == RET_PATH_TC && !bp.core.ring && D % tcg::BK == 0 && (H * d_k) % tcg::BN == 0 &&
          (H * d_v) % tcg::BN == 0 && (H * d_v) % tcg::BK == 0 && D_out % tcg::BN == 0 && d_v % 8 == 0;
  const size_t M = static_cast<size_t>(B) * L, HV = static_cast<size_t>(H) * d_v;
  size_t off = bp.core.bytes;
  bp.off_cs = off; off += up256(static_cast<size_t>(L) * (d_k / 2) * 8);
  bp.off_v = off; off += up256(M * HV * 2);
  bp.off_o = off; off += up256(M * HV * 4);
  bp.off_g = off; off += up256(M * HV * 2);
  bp.off_a = off; off += up256(M * HV * 2);
  bp.bytes = off;
  return bp;
}

// C = A·W on the pair GEMM kernel; A [M][K] bf16, W [K][N] bf16.
template <int MODE>
cudaError_t launch_gemm(const void* A, int M, int K, const void* W, int N, tcg::GemmArgs g,
                        const CallConsts& cc, cudaStream_t st, const char* name) {
  CUtensorMap ma, mw;
  if (!make_map(&ma, A, static_cast<uint64_t>(M), static_cast<uint64_t>(K)) ||
      !make_map(&mw, W, static_cast<uint64_t>(K), static_cast<uint64_t>(N), 64))
    return cudaErrorInvalidValue;
  g.M = M;
  g.N = N;
  g.K = K;
  cudaError_t e = cudaFuncSetAttribute(tcg::proj_gemm_kernel<MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tcg::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ((M + 2 * tcg::BM - 1) / (2 * tcg::BM)), N / tcg::BN);
  cfg.blockDim = dim3(tcg::NTHREADS);
  cfg.dynamicSmemBytes = tcg::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  Mark m(name, st);
  e = cudaLaunchKernelEx(&cfg, tcg::proj_gemm_kernel<MODE>, ma, mw, g, cc);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Scratch of ret_chunkwise_noalloc: part of this module's device image, so
// using it allocates nothing at call time.  In host code the array's name is
// only a stand-in; its device address comes from cudaGetSymbolAddress with
// the caller's device current.  The lookup is repeated on every call made
// outside stream capture, so a device reset or a re-created primary context
// (which reloads the module and may move the array) never leaves a stale
// address behind.  A call made while its stream is capturing reuses the
// address that the last uncaptured call on that device found (the lookup may
// have to load the module, which does not belong inside a capture).
__device__ __align__(256) unsigned char g_noalloc_scratch[RET_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

ret_status noalloc_scratch(cudaStream_t stream, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return RET_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return RET_EUNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return RET_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (cap == cudaStreamCaptureStatusNone || !g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return RET_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return RET_OK;
}

}  // namespace

// ===========================================================================
// Exported entry points
// ===========================================================================
extern "C" {

const char* ret_status_string(ret_status s) {
  switch (s) {
    case RET_OK: return "ok";
    case RET_EINVAL: return "invalid argument";
    case RET_EUNSUPPORTED: return "arguments outside the implemented domain";
    case RET_ECUDA: return "CUDA error";
    case RET_ETIMEOUT: return "a kernel's bounded wait expired";
    case RET_EWORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

int ret_abi_version(void) { return RET_ABI_VERSION; }

ret_status ret_profile_begin(cudaEvent_t* events, int n_events) {
  if (!events || n_events < 2) return RET_EINVAL;
  g_prof.ev = events;
  g_prof.cap = n_events;
  g_prof.used = 0;
  return RET_OK;
}

int ret_profile_end(void) {
  const int n = g_prof.used;
  g_prof.ev = nullptr;
  g_prof.cap = 0;
  return n;
}

const char* ret_profile_kernel(int i) {
  return (i >= 0 && i < g_prof.used && i < 64) ? g_prof.names[i] : "";
}

ret_status ret_force_path(int path) {
  if (path != 0 && path != RET_PATH_SIMT && path != RET_PATH_TC && path != RET_PATH_TC_SINGLE &&
      path != RET_PATH_TC_CARRY)
    return RET_EINVAL;
  g_force_path = path;
  return RET_OK;
}

int ret_chunk_size(ret_dtype in_dt, const float* gamma, int H, int L, int d_k, int d_v) {
  if (in_dt != RET_F32 && in_dt != RET_BF16) return 0;
  if (H < 1 || H > kMaxHeads || L < 1 || d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) || d_v < 1 ||
      d_v > 1024)
    return 0;
  if (gamma)
    for (int h = 0; h < H; ++h)
      if (!(gamma[h] > 0.f) || !(gamma[h] <= 1.f)) return 0;
  if (tc_chunk_ok(in_dt, gamma, H, L, d_k, d_v, tcc::CH)) return tcc::CH;
  const long long b = std::llround(std::sqrt(static_cast<double>(L)));
  return static_cast<int>(std::max(1LL, std::min<long long>(b, L)));
}

ret_status ret_chunkwise_plan(ret_dtype in_dt, const float* gamma, int B, int H, int L, int d_k,
                              int d_v, int chunk, ret_dtype out_dt, int gn_enabled, int* path,
                              size_t* workspace_bytes) {
  if (!path || !workspace_bytes) return RET_EINVAL;
  if (in_dt != RET_F32 && in_dt != RET_BF16) return RET_EINVAL;
  if (out_dt != RET_F32 && out_dt != RET_BF16) return RET_EINVAL;
  if (B < 1 || H < 1 || H > kMaxHeads || L < 1 || d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) ||
      d_v < 1 || d_v > 1024 || chunk < 1)
    return RET_EINVAL;
  const Plan p = plan_chunkwise(in_dt, gamma, B, H, L, d_k, d_v, chunk, gn_enabled != 0);
  *path = p.path;
  *workspace_bytes = p.bytes;
  return RET_OK;
}

ret_status ret_chunkwise_plan_compact(ret_dtype in_dt, const float* gamma, int B, int H, int L,
                                      int d_k, int d_v, int chunk, ret_dtype out_dt, int gn_enabled,
                                      int* path, size_t* workspace_bytes) {
  if (!path || !workspace_bytes) return RET_EINVAL;
  if (in_dt != RET_F32 && in_dt != RET_BF16) return RET_EINVAL;
  if (out_dt != RET_F32 && out_dt != RET_BF16) return RET_EINVAL;
  if (B < 1 || H < 1 || H > kMaxHeads || L < 1 || d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) ||
      d_v < 1 || d_v > 1024 || chunk < 1)
    return RET_EINVAL;
  const Plan p = plan_chunkwise(in_dt, gamma, B, H, L, d_k, d_v, chunk, gn_enabled != 0);
  const Plan pc = plan_chunkwise(in_dt, gamma, B, H, L, d_k, d_v, chunk, gn_enabled != 0, false, true);
  const Plan& best = pc.bytes < p.bytes ? pc : p;   // the compact mode only where it is smaller
  *path = best.path;
  *workspace_bytes = best.bytes;
  return RET_OK;
}

}  // extern "C"

namespace {
// Shared body of ret_chunkwise (scan = false) and ret_chunkwise_scan (true).
ret_status chunkwise_impl(const void* q, const void* k, const void* v, ret_dtype in_dt,
                          const float* gamma, const float* theta, int B, int H, int L, int d_k,
                          int d_v, int64_t pos0, int chunk, const float* state_in,
                          float* state_out, void* out, ret_dtype out_dt, const ret_gn* gn,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream,
                          bool scan, const int64_t* row_pos0 = nullptr) {
  ret_status s = check_common(q, k, v, in_dt, B, H, L, d_k, d_v, pos0, state_in, state_out, out,
                              out_dt, gn);
  if (s != RET_OK) return s;
  RowPos rp = no_rowpos();
  if (row_pos0) {   // one start position per batch row
    if (B > kMaxRowPos) return RET_EUNSUPPORTED;
    for (int b = 0; b < B; ++b) {
      if (row_pos0[b] < 0 || row_pos0[b] + L > kMaxPos) return RET_EINVAL;
      rp.p[b] = static_cast<float>(row_pos0[b]);
    }
    rp.on = 1;
  }
  if (chunk < 1) return RET_EINVAL;
  if (!gamma || !theta) return RET_EINVAL;
  Plan p = plan_chunkwise(in_dt, gamma, B, H, L, d_k, d_v, chunk, gn_on(gn), scan);
  if (p.bytes > 0 && workspace && al16(workspace) && workspace_bytes < p.bytes && !scan) {
    // too short for the front pass: the compact-workspace mode, where it applies
    const Plan pc = plan_chunkwise(in_dt, gamma, B, H, L, d_k, d_v, chunk, gn_on(gn), false, true);
    if (pc.ring && workspace_bytes >= pc.bytes) p = pc;
  }
  // γ^b of the chunks: the 128-token tile on the tensor-core path
  CallConsts cc;
  if ((s = make_consts(cc, gamma, theta, H, d_k, p.path == RET_PATH_TC ? tcc::CH : chunk, L)) != RET_OK)
    return s;
  if (p.bytes > 0 && (!workspace || workspace_bytes < p.bytes || !al16(workspace)))
    return RET_EWORKSPACE;
  if (p.path == RET_PATH_TC) {
    const auto* qq = static_cast<const __nv_bfloat16*>(q);
    const auto* kk = static_cast<const __nv_bfloat16*>(k);
    const auto* vv = static_cast<const __nv_bfloat16*>(v);
    const bool sc = scan || p.scan;
    if (out_dt == RET_F32)
      return run_tc_chunk<float>(qq, kk, vv, cc, B, H, L, d_k, d_v, pos0, state_in, state_out,
                                 static_cast<float*>(out), gn, workspace, p, stream, rp, sc);
    return run_tc_chunk<__nv_bfloat16>(qq, kk, vv, cc, B, H, L, d_k, d_v, pos0, state_in,
                                       state_out, static_cast<__nv_bfloat16*>(out), gn, workspace,
                                       p, stream, rp, sc);
  }
  // The fp32 kernels always run in the chunk-parallel layout.
  if (in_dt == RET_F32)
    return dispatch_simt_out<float>(q, k, v, cc, B, H, L, d_k, d_v, pos0, chunk, state_in,
                                    state_out, out, out_dt, gn, workspace, p, true, stream, rp);
  return dispatch_simt_out<__nv_bfloat16>(q, k, v, cc, B, H, L, d_k, d_v, pos0, chunk, state_in,
                                          state_out, out, out_dt, gn, workspace, p, true, stream,
                                          rp);
}
}  // namespace

extern "C" {

ret_status ret_chunkwise(const void* q, const void* k, const void* v, ret_dtype in_dt,
                         const float* gamma, const float* theta, int B, int H, int L, int d_k,
                         int d_v, int64_t pos0, int chunk, const float* state_in,
                         float* state_out, void* out, ret_dtype out_dt, const ret_gn* gn,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Range nv("ret_chunkwise");
  return chunkwise_impl(q, k, v, in_dt, gamma, theta, B, H, L, d_k, d_v, pos0, chunk, state_in,
                        state_out, out, out_dt, gn, workspace, workspace_bytes, stream, false);
}

ret_status ret_chunkwise_rowpos(const void* q, const void* k, const void* v, ret_dtype in_dt,
                                const float* gamma, const float* theta, int B, int H, int L,
                                int d_k, int d_v, const int64_t* row_pos0, int chunk,
                                const float* state_in, float* state_out, void* out,
                                ret_dtype out_dt, const ret_gn* gn, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  Range nv("ret_chunkwise_rowpos");
  if (!row_pos0) return RET_EINVAL;
  return chunkwise_impl(q, k, v, in_dt, gamma, theta, B, H, L, d_k, d_v, 0, chunk, state_in,
                        state_out, out, out_dt, gn, workspace, workspace_bytes, stream, false,
                        row_pos0);
}

ret_status ret_chunkwise_noalloc(const void* q, const void* k, const void* v, ret_dtype in_dt,
                                 const float* gamma, const float* theta, int B, int H, int L,
                                 int d_k, int d_v, int64_t pos0, int chunk,
                                 const float* state_in, float* state_out, void* out,
                                 ret_dtype out_dt, const ret_gn* gn, cudaStream_t stream) {
  Range nv("ret_chunkwise_noalloc");
  ret_status s = check_common(q, k, v, in_dt, B, H, L, d_k, d_v, pos0, state_in, state_out, out,
                              out_dt, gn);
  if (s != RET_OK) return s;
  if (chunk < 1) return RET_EINVAL;
  const Plan p = plan_chunkwise(in_dt, gamma, B, H, L, d_k, d_v, chunk, gn_on(gn));
  const Plan pc = plan_chunkwise(in_dt, gamma, B, H, L, d_k, d_v, chunk, gn_on(gn), false, true);
  if (p.bytes > static_cast<size_t>(RET_NOALLOC_SCRATCH_BYTES) &&
      pc.bytes > static_cast<size_t>(RET_NOALLOC_SCRATCH_BYTES))
    return RET_EWORKSPACE;
  void* scratch = nullptr;
  if ((s = noalloc_scratch(stream, &scratch)) != RET_OK) return s;
  return ret_chunkwise(q, k, v, in_dt, gamma, theta, B, H, L, d_k, d_v, pos0, chunk, state_in,
                       state_out, out, out_dt, gn, scratch, RET_NOALLOC_SCRATCH_BYTES, stream);
}

ret_status ret_chunkwise_scan_plan(ret_dtype in_dt, const float* gamma, int B, int H, int L,
                                   int d_k, int d_v, int chunk, ret_dtype out_dt, int gn_enabled,
                                   int* path, size_t* workspace_bytes) {
  if (!path || !workspace_bytes) return RET_EINVAL;
  if (in_dt != RET_F32 && in_dt != RET_BF16) return RET_EINVAL;
  if (out_dt != RET_F32 && out_dt != RET_BF16) return RET_EINVAL;
  if (B < 1 || H < 1 || H > kMaxHeads || L < 1 || d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) ||
      d_v < 1 || d_v > 1024 || chunk < 1)
    return RET_EINVAL;
  const Plan p = plan_chunkwise(in_dt, gamma, B, H, L, d_k, d_v, chunk, gn_enabled != 0, true);
  *path = p.path;
  *workspace_bytes = p.bytes;
  return RET_OK;
}

ret_status ret_chunkwise_scan(const void* q, const void* k, const void* v, ret_dtype in_dt,
                              const float* gamma, const float* theta, int B, int H, int L,
                              int d_k, int d_v, int64_t pos0, int chunk, const float* state_in,
                              float* state_out, void* out, ret_dtype out_dt, const ret_gn* gn,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Range nv("ret_chunkwise_scan");
  return chunkwise_impl(q, k, v, in_dt, gamma, theta, B, H, L, d_k, d_v, pos0, chunk, state_in,
                        state_out, out, out_dt, gn, workspace, workspace_bytes, stream, true);
}

ret_status ret_chunkwise_backward_plan(ret_dtype in_dt, const float* gamma, int B, int H, int L,
                                       int d_k, int d_v, int chunk, int* path,
                                       size_t* workspace_bytes) {
  if (!path || !workspace_bytes) return RET_EINVAL;
  if (in_dt != RET_F32 && in_dt != RET_BF16) return RET_EINVAL;
  if (B < 1 || H < 1 || H > kMaxHeads || L < 1 || d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) ||
      d_v < 1 || d_v > 1024 || chunk < 1)
    return RET_EINVAL;
  if (tc_backward_ok(in_dt, gamma, H, d_k, d_v, chunk, B)) {
    *path = RET_PATH_TC;
    *workspace_bytes = plan_tc_backward(B, H, L, d_k, d_v).bytes;
  } else {
    *path = RET_PATH_SIMT;
    *workspace_bytes = plan_backward(in_dt, B, H, L, d_k, d_v, chunk).bytes;
  }
  return RET_OK;
}

ret_status ret_chunkwise_backward(const void* q, const void* k, const void* v, const void* d_out,
                                  ret_dtype in_dt, const float* gamma, const float* theta, int B,
                                  int H, int L, int d_k, int d_v, int64_t pos0, int chunk,
                                  const float* state_in, const float* d_state_out, void* dq,
                                  void* dk, void* dv, ret_dtype grad_dt, float* d_state_in,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Range nv("ret_chunkwise_backward");
  ret_status s = check_common(q, k, v, in_dt, B, H, L, d_k, d_v, pos0, state_in, d_state_in, dq,
                              grad_dt, nullptr);
  if (s != RET_OK) return s;
  if (!d_out || !dk || !dv || !al16(d_out) || !al16(dk) || !al16(dv)) return RET_EINVAL;
  if (d_state_out && !al16(d_state_out)) return RET_EINVAL;
  if (chunk < 1) return RET_EINVAL;
  const int64_t nch = (static_cast<int64_t>(L) + chunk - 1) / chunk;
  if (static_cast<int64_t>(B) * H > 65535) return RET_EUNSUPPORTED;   // state tiles: one grid.z row per head
  CallConsts cc;
  if ((s = make_consts(cc, gamma, theta, H, d_k, chunk, L)) != RET_OK) return s;
  for (int h = 0; h < H; ++h)   // the reversed evaluations start from dS_out/γ
    if (gamma[h] < 0x1p-64f) return RET_EUNSUPPORTED;
  if (tc_backward_ok(in_dt, gamma, H, d_k, d_v, chunk, B)) {
    const TcBwdPlan tp = plan_tc_backward(B, H, L, d_k, d_v);
    if (!workspace || workspace_bytes < tp.bytes || !al16(workspace)) return RET_EWORKSPACE;
    const auto* a = static_cast<const __nv_bfloat16*>(q);
    const auto* b = static_cast<const __nv_bfloat16*>(k);
    const auto* c = static_cast<const __nv_bfloat16*>(v);
    const auto* d = static_cast<const __nv_bfloat16*>(d_out);
    if (grad_dt == RET_F32)
      return run_tc_backward<float>(a, b, c, d, cc, B, H, L, d_k, d_v, pos0, state_in, d_state_out,
                                    static_cast<float*>(dq), static_cast<float*>(dk),
                                    static_cast<float*>(dv), d_state_in, workspace, tp, stream);
    return run_tc_backward<__nv_bfloat16>(a, b, c, d, cc, B, H, L, d_k, d_v, pos0, state_in,
                                          d_state_out, static_cast<__nv_bfloat16*>(dq),
                                          static_cast<__nv_bfloat16*>(dk),
                                          static_cast<__nv_bfloat16*>(dv), d_state_in, workspace,
                                          tp, stream);
  }
  const BwdPlan p = plan_backward(in_dt, B, H, L, d_k, d_v, chunk);
  if (!workspace || workspace_bytes < p.bytes || !al16(workspace)) return RET_EWORKSPACE;
  if (in_dt == RET_F32) {
    const auto* a = static_cast<const float*>(q);
    const auto* b = static_cast<const float*>(k);
    const auto* c = static_cast<const float*>(v);
    const auto* d = static_cast<const float*>(d_out);
    if (grad_dt == RET_F32)
      return run_backward<float, float>(a, b, c, d, cc, B, H, L, d_k, d_v, pos0, chunk, state_in,
                                        d_state_out, static_cast<float*>(dq),
                                        static_cast<float*>(dk), static_cast<float*>(dv),
                                        d_state_in, workspace, p, stream);
    return run_backward<float, __nv_bfloat16>(
        a, b, c, d, cc, B, H, L, d_k, d_v, pos0, chunk, state_in, d_state_out,
        static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk),
        static_cast<__nv_bfloat16*>(dv), d_state_in, workspace, p, stream);
  }
  const auto* a = static_cast<const __nv_bfloat16*>(q);
  const auto* b = static_cast<const __nv_bfloat16*>(k);
  const auto* c = static_cast<const __nv_bfloat16*>(v);
  const auto* d = static_cast<const __nv_bfloat16*>(d_out);
  if (grad_dt == RET_F32)
    return run_backward<__nv_bfloat16, float>(a, b, c, d, cc, B, H, L, d_k, d_v, pos0, chunk,
                                              state_in, d_state_out, static_cast<float*>(dq),
                                              static_cast<float*>(dk), static_cast<float*>(dv),
                                              d_state_in, workspace, p, stream);
  return run_backward<__nv_bfloat16, __nv_bfloat16>(
      a, b, c, d, cc, B, H, L, d_k, d_v, pos0, chunk, state_in, d_state_out,
      static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk),
      static_cast<__nv_bfloat16*>(dv), d_state_in, workspace, p, stream);
}

ret_status ret_parallel_plan(ret_dtype in_dt, const float* gamma, int B, int H, int L, int d_k,
                             int d_v, ret_dtype out_dt, int gn_enabled, int state_out_wanted,
                             int* path, size_t* workspace_bytes) {
  if (!path || !workspace_bytes) return RET_EINVAL;
  if (in_dt != RET_F32 && in_dt != RET_BF16) return RET_EINVAL;
  if (out_dt != RET_F32 && out_dt != RET_BF16) return RET_EINVAL;
  if (B < 1 || H < 1 || H > kMaxHeads || L < 1 || d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) ||
      d_v < 1 || d_v > 1024)
    return RET_EINVAL;
  const Plan p = plan_parallel(in_dt, gamma, B, H, L, d_k, d_v, gn_enabled != 0, state_out_wanted != 0);
  *path = p.path;
  *workspace_bytes = p.bytes;
  return RET_OK;
}

ret_status ret_parallel(const void* q, const void* k, const void* v, ret_dtype in_dt,
                        const float* gamma, const float* theta, int B, int H, int L, int d_k,
                        int d_v, int64_t pos0, const float* state_in, float* state_out,
                        void* out, ret_dtype out_dt, const ret_gn* gn, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  Range nv("ret_parallel");
  ret_status s = check_common(q, k, v, in_dt, B, H, L, d_k, d_v, pos0, state_in, state_out, out,
                              out_dt, gn);
  if (s != RET_OK) return s;
  CallConsts cc;
  const Plan p = plan_parallel(in_dt, gamma, B, H, L, d_k, d_v, gn_on(gn), state_out != nullptr);
  if (!workspace || workspace_bytes < p.bytes || !al16(workspace)) return RET_EWORKSPACE;
  if (p.path == RET_PATH_TC) {
    // 128-row blocks (the front pass folds ζ over blocks of 128)
    if ((s = make_consts(cc, gamma, theta, H, d_k, tcc::CH, L)) != RET_OK) return s;
    const auto* qq = static_cast<const __nv_bfloat16*>(q);
    const auto* kk = static_cast<const __nv_bfloat16*>(k);
    const auto* vv = static_cast<const __nv_bfloat16*>(v);
    if (out_dt == RET_F32)
      return run_tc_chunk<float>(qq, kk, vv, cc, B, H, L, d_k, d_v, pos0, state_in, state_out,
                                 static_cast<float*>(out), gn, workspace, p, stream, no_rowpos(),
                                 false, true);
    return run_tc_chunk<__nv_bfloat16>(qq, kk, vv, cc, B, H, L, d_k, d_v, pos0, state_in,
                                       state_out, static_cast<__nv_bfloat16*>(out), gn, workspace,
                                       p, stream, no_rowpos(), false, true);
  }
  if ((s = make_consts(cc, gamma, theta, H, d_k, L, L)) != RET_OK) return s;
  // One chunk of length L: the fp32 chunk kernels evaluate the parallel form.
  if (in_dt == RET_F32)
    return dispatch_simt_out<float>(q, k, v, cc, B, H, L, d_k, d_v, pos0, L, state_in, state_out,
                                    out, out_dt, gn, workspace, p, state_out != nullptr, stream,
                                    no_rowpos());
  return dispatch_simt_out<__nv_bfloat16>(q, k, v, cc, B, H, L, d_k, d_v, pos0, L, state_in,
                                          state_out, out, out_dt, gn, workspace, p,
                                          state_out != nullptr, stream, no_rowpos());
}

ret_status ret_step(const void* q, const void* k, const void* v, ret_dtype in_dt,
                    const float* gamma, const float* theta, int B, int H, int d_k, int d_v,
                    int64_t pos, float* state, void* out, ret_dtype out_dt, const ret_gn* gn,
                    cudaStream_t stream) {
  Range nv("ret_step");
  ret_status s = check_common(q, k, v, in_dt, B, H, 1, d_k, d_v, pos, state, state, out, out_dt, gn);
  if (s != RET_OK) return s;
  if (!state) return RET_EINVAL;
  CallConsts cc;
  if ((s = make_consts(cc, gamma, theta, H, d_k, 1, 1)) != RET_OK) return s;
  const int vec = (d_v % 4 == 0) ? 4 : 1;
  const int threads = (d_v + vec - 1) / vec;
  if (threads > 256) return RET_EUNSUPPORTED;
  const int nthr = ((threads + 31) / 32) * 32;
  const size_t smem = (2 * static_cast<size_t>(d_k) + 64) * sizeof(float);
  const int BH = B * H;
  const int g = gn_on(gn) ? 1 : 0;
  const float eps = g ? gn->eps : 0.f;
  const float* gw = g ? gn->weight : nullptr;
  const float* gbb = g ? gn->bias : nullptr;
  const float fpos = static_cast<float>(pos);
  Mark mark("decode_step", stream);
#define RET_DECODE(TIN, TOUT, VEC)                                                           \
  simt::decode_step_kernel<TIN, TOUT, VEC><<<BH, nthr, smem, stream>>>(                      \
      static_cast<const TIN*>(q), static_cast<const TIN*>(k), static_cast<const TIN*>(v),     \
      state, static_cast<TOUT*>(out), cc, H, d_k, d_v, fpos, g, eps, gw, gbb)
  if (in_dt == RET_BF16) {
    if (out_dt == RET_BF16) { if (vec == 4) RET_DECODE(__nv_bfloat16, __nv_bfloat16, 4); else RET_DECODE(__nv_bfloat16, __nv_bfloat16, 1); }
    else { if (vec == 4) RET_DECODE(__nv_bfloat16, float, 4); else RET_DECODE(__nv_bfloat16, float, 1); }
  } else {
    if (out_dt == RET_BF16) { if (vec == 4) RET_DECODE(float, __nv_bfloat16, 4); else RET_DECODE(float, __nv_bfloat16, 1); }
    else { if (vec == 4) RET_DECODE(float, float, 4); else RET_DECODE(float, float, 1); }
  }
#undef RET_DECODE
  return last_launch();
}

ret_status ret_rotate(const void* x, ret_dtype in_dt, const float* theta, int B, int H, int L,
                      int d, int64_t pos0, float scale, void* y, ret_dtype out_dt,
                      cudaStream_t stream) {
  Range nv("ret_rotate");
  if (!x || !y || !theta || !al16(x) || !al16(y)) return RET_EINVAL;
  if (in_dt != RET_F32 && in_dt != RET_BF16) return RET_EINVAL;
  if (out_dt != RET_F32 && out_dt != RET_BF16) return RET_EINVAL;
  if (B < 1 || H < 1 || L < 1 || d < 2 || d > 2 * kMaxPairs || (d & 1)) return RET_EINVAL;
  if (pos0 < 0 || pos0 + L > kMaxPos || !std::isfinite(scale)) return RET_EINVAL;
  CallConsts cc;
  std::memset(&cc, 0, sizeof(cc));
  for (int i = 0; i < d / 2; ++i) {
    if (!std::isfinite(theta[i])) return RET_EINVAL;
    cc.theta[i] = theta[i];
  }
  const int BH = B * H;
  const dim3 grid = fold_y((d / 2 + 31) / 32, (static_cast<size_t>(L) + 7) / 8);
  const float p0 = static_cast<float>(pos0);
  if (in_dt == RET_BF16 && out_dt == RET_BF16)
    simt::rotate_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, dim3(32, 8), 0, stream>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), cc, BH, H, L, d, p0, scale, no_rowpos(), 0);
  else if (in_dt == RET_BF16)
    simt::rotate_kernel<__nv_bfloat16, float><<<grid, dim3(32, 8), 0, stream>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<float*>(y), cc, BH, H, L, d, p0, scale, no_rowpos(), 0);
  else if (out_dt == RET_BF16)
    simt::rotate_kernel<float, __nv_bfloat16><<<grid, dim3(32, 8), 0, stream>>>(
        static_cast<const float*>(x), static_cast<__nv_bfloat16*>(y), cc, BH, H, L, d, p0, scale, no_rowpos(), 0);
  else
    simt::rotate_kernel<float, float><<<grid, dim3(32, 8), 0, stream>>>(
        static_cast<const float*>(x), static_cast<float*>(y), cc, BH, H, L, d, p0, scale, no_rowpos(), 0);
  return last_launch();
}

ret_status ret_decay_row_norm(void* out, ret_dtype out_dt, const float* gamma, int B, int H,
                              int L, int d_v, int64_t pos0, cudaStream_t stream) {
  Range nv("ret_decay_row_norm");
  if (!out || !al16(out) || (out_dt != RET_F32 && out_dt != RET_BF16)) return RET_EINVAL;
  if (B < 1 || H < 1 || H > kMaxHeads || L < 1 || d_v < 1 || d_v > 1024) return RET_EINVAL;
  if (pos0 < 0 || pos0 + L > kMaxPos) return RET_EINVAL;
  const int64_t rows = static_cast<int64_t>(B) * H * L;
  if (rows >= (int64_t(1) << 31)) return RET_EINVAL;
  if (!gamma) return RET_EINVAL;
  CallConsts cc;
  std::memset(&cc, 0, sizeof(cc));
  for (int h = 0; h < H; ++h) {
    if (!(gamma[h] > 0.f) || !(gamma[h] <= 1.f)) return RET_EINVAL;
    cc.lg2g[h] = static_cast<float>(std::log2(static_cast<double>(gamma[h])));
  }
  Mark m("decay_row_norm", stream);
  const int esz = out_dt == RET_F32 ? 4 : 2;
  if ((static_cast<size_t>(d_v) * esz) % 16 == 0) {   // whole 16-byte vectors per row
    const int vpr = d_v * esz / 16;
    const size_t groups = (static_cast<size_t>(rows) + 31) / 32;
    const unsigned grid = static_cast<unsigned>(std::min<size_t>((groups + 7) / 8, 148 * 8));
    if (out_dt == RET_F32)
      simt::decay_row_norm_vec_kernel<float><<<grid, 256, 0, stream>>>(
          static_cast<uint4*>(out), cc, H, L, vpr, static_cast<size_t>(rows), static_cast<float>(pos0));
    else
      simt::decay_row_norm_vec_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
          static_cast<uint4*>(out), cc, H, L, vpr, static_cast<size_t>(rows), static_cast<float>(pos0));
    return last_launch();
  }
  if (out_dt == RET_F32)
    simt::decay_row_norm_kernel<float><<<static_cast<unsigned>(rows), 128, 0, stream>>>(
        static_cast<float*>(out), cc, H, L, d_v, static_cast<float>(pos0));
  else
    simt::decay_row_norm_kernel<__nv_bfloat16><<<static_cast<unsigned>(rows), 128, 0, stream>>>(
        static_cast<__nv_bfloat16*>(out), cc, H, L, d_v, static_cast<float>(pos0));
  return last_launch();
}

ret_status ret_matmul(const void* a, const void* w, void* c, ret_dtype c_dt, int M, int N, int K,
                      cudaStream_t stream) {
  Range nv("ret_matmul");
  if (!a || !w || !c || !al16(a) || !al16(w) || !al16(c)) return RET_EINVAL;
  if (c_dt != RET_F32 && c_dt != RET_BF16) return RET_EINVAL;
  if (M < 1 || N < 1 || K < 1) return RET_EINVAL;
  if (N % tcg::BN != 0 || K % tcg::BK != 0) return RET_EUNSUPPORTED;
  CallConsts cc;
  std::memset(&cc, 0, sizeof(cc));
  tcg::GemmArgs g;
  g.out = c;
  g.out_f32 = c_dt == RET_F32 ? 1 : 0;
  return launch_gemm<tcg::PLAIN>(a, M, K, w, N, g, cc, stream, "matmul") == cudaSuccess ? RET_OK : RET_ECUDA;
}

ret_status ret_msr_block_plan(const float* gamma, int B, int L, int D, int H, int d_k, int d_v,
                              int D_out, size_t* workspace_bytes) {
  if (!workspace_bytes) return RET_EINVAL;
  if (B < 1 || L < 1 || D < 1 || H < 1 || H > kMaxHeads || d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) ||
      d_v < 1 || d_v > 1024 || D_out < 1)
    return RET_EINVAL;
  const BlockPlan bp = plan_block(gamma, B, L, D, H, d_k, d_v, D_out);
  if (!bp.ok) return RET_EUNSUPPORTED;
  *workspace_bytes = bp.bytes;
  return RET_OK;
}

ret_status ret_msr_block(const void* x, const void* w_q, const void* w_k, const void* w_v,
                         const void* w_g, const void* w_o, const float* gamma, const float* theta,
                         int B, int L, int D, int H, int d_k, int d_v, int D_out, int64_t pos0,
                         const float* state_in, float* state_out, void* z, ret_dtype z_dt,
                         float gn_eps, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Range nv("ret_msr_block");
  if (!x || !w_q || !w_k || !w_v || !w_g || !w_o || !z) return RET_EINVAL;
  for (const void* ptr : {x, w_q, w_k, w_v, w_g, w_o, static_cast<const void*>(z)})
    if (!al16(ptr)) return RET_EINVAL;
  if ((state_in && !al16(state_in)) || (state_out && !al16(state_out))) return RET_EINVAL;
  if (z_dt != RET_F32 && z_dt != RET_BF16) return RET_EINVAL;
  if (B < 1 || L < 1 || D < 1 || H < 1 || H > kMaxHeads || d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) ||
      d_v < 1 || d_v > 1024 || D_out < 1)
    return RET_EINVAL;
  if (pos0 < 0 || pos0 + L > kMaxPos || static_cast<int64_t>(B) * H * L >= (int64_t(1) << 31)) return RET_EINVAL;
  if (!(gn_eps > 0.f) || !std::isfinite(gn_eps)) return RET_EINVAL;
  CallConsts cc;
  ret_status s;
  if ((s = make_consts(cc, gamma, theta, H, d_k, tcc::CH, L)) != RET_OK) return s;
  const BlockPlan bp = plan_block(gamma, B, L, D, H, d_k, d_v, D_out);
  if (!bp.ok) return RET_EUNSUPPORTED;
  if (!workspace || workspace_bytes < bp.bytes || !al16(workspace)) return RET_EWORKSPACE;
  const int M = B * L, HK = H * d_k, HV = H * d_v;
  const int Lp = ((L + tcc::CH - 1) / tcc::CH) * tcc::CH;
  auto* qr = wsp<__nv_bfloat16>(workspace, bp.core.off_q);
  auto* kr = wsp<__nv_bfloat16>(workspace, bp.core.off_k);
  auto* cs = wsp<float2>(workspace, bp.off_cs);
  auto* vh = wsp<__nv_bfloat16>(workspace, bp.off_v);
  auto* of = wsp<float>(workspace, bp.off_o);
  auto* gt = wsp<__nv_bfloat16>(workspace, bp.off_g);
  auto* ao = wsp<__nv_bfloat16>(workspace, bp.off_a);
  {
    const size_t n = static_cast<size_t>(L) * (d_k / 2);
    Mark m("angle_table", stream);
    tcc::angle_table_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
        cs, cc, L, d_k / 2, static_cast<float>(pos0));
    if (cudaGetLastError() != cudaSuccess) return RET_ECUDA;
  }
  tcg::GemmArgs g;
  g.L = L;
  g.Lp = Lp;
  g.H = H;
  g.dh = d_k;
  g.pos0 = static_cast<float>(pos0);
  g.cs = cs;
  g.out = qr;   // q = x·W_Q → Q″ (rotated, ω folded)
  if (launch_gemm<tcg::ROT_Q>(x, M, D, w_q, HK, g, cc, stream, "proj_q_rot") != cudaSuccess) return RET_ECUDA;
  g.out = kr;   // k = x·W_K → K̂′ (rotated, d_k^{-1/2}·ζ folded)
  if (launch_gemm<tcg::ROT_K>(x, M, D, w_k, HK, g, cc, stream, "proj_k_rot") != cudaSuccess) return RET_ECUDA;
  if (Lp > L) {   // the zero rows that pad every sequence to whole chunks
    const size_t pitch = static_cast<size_t>(Lp) * d_k * 2, width = static_cast<size_t>(Lp - L) * d_k * 2;
    const size_t start = static_cast<size_t>(L) * d_k;
    if (cudaMemset2DAsync(qr + start, pitch, 0, width, static_cast<size_t>(B) * H, stream) != cudaSuccess ||
        cudaMemset2DAsync(kr + start, pitch, 0, width, static_cast<size_t>(B) * H, stream) != cudaSuccess)
      return RET_ECUDA;
  }
  g.out = vh;   // v = x·W_V, per head
  g.dh = d_v;
  if (launch_gemm<tcg::HEADS>(x, M, D, w_v, HV, g, cc, stream, "proj_v") != cudaSuccess) return RET_ECUDA;
  // the chunkwise core on the projected operands, fp32 output for GroupNorm
  if ((s = run_tc_chunk<float>(nullptr, nullptr, vh, cc, B, H, L, d_k, d_v, pos0, state_in, state_out, of,
                               nullptr, workspace, bp.core, stream, no_rowpos(), bp.core.scan, false,
                               true)) != RET_OK)
    return s;
  tcg::GemmArgs gp;
  gp.out = gt;   // the gate's pre-activation x·W_G
  if (launch_gemm<tcg::PLAIN>(x, M, D, w_g, HV, gp, cc, stream, "proj_gate") != cudaSuccess) return RET_ECUDA;
  {
    const size_t rows = static_cast<size_t>(B) * H * L;
    Mark m("gn_gate", stream);
    tcg::gn_gate_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(of, gt, ao, H, L, d_v, rows,
                                                                                    gn_eps);
    if (cudaGetLastError() != cudaSuccess) return RET_ECUDA;
  }
  gp.out = z;   // z = (swish(x·W_G) ⊙ GN(O))·W_O
  gp.out_f32 = z_dt == RET_F32 ? 1 : 0;
  if (launch_gemm<tcg::PLAIN>(ao, M, HV, w_o, D_out, gp, cc, stream, "proj_out") != cudaSuccess) return RET_ECUDA;
  return last_launch();
}

}  // extern "C"

namespace {
// ---------------------------------------------------------------------------
// Parameter gradients and GroupNorm backward: workspace layouts and launches
// ---------------------------------------------------------------------------
struct ParamPlan {
  int nseg, C, ntk, ntv, Lp;
  bool fast;     // d_k, d_v multiples of 64: prepped fp32 operands, 64-thread walks
  bool tc_ok;    // d_k, d_v multiples of 128: the tensor-core walks (bf16 inputs)
  size_t off_g, off_t, off_cs, off_states, off_gw, off_z, off_qb, off_kf, bytes;
};

ParamPlan plan_param_grads(int B, int H, int L, int d_k, int d_v) {
  ParamPlan p{};
  p.nseg = (L + grad::kRowsPerBlock - 1) / grad::kRowsPerBlock;
  p.C = (L + grad::kGradChunk - 1) / grad::kGradChunk;
  p.ntk = (d_k + grad::kTile - 1) / grad::kTile;
  p.ntv = (d_v + grad::kTile - 1) / grad::kTile;
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t nblk = BH * p.nseg, nwalk = BH * p.ntk * p.ntv;
  size_t off = 0;
  p.off_g = off; off += up256(nblk * sizeof(double));
  p.off_t = off; off += up256(nblk * static_cast<size_t>(d_k / 2) * sizeof(float));
  p.off_cs = off; off += up256(static_cast<size_t>(L) * (d_k / 2) * sizeof(float2));
  p.off_states = off; off += up256(nwalk * p.C * 4096 * sizeof(float));
  p.off_gw = off; off += up256(nwalk * sizeof(double));
  p.off_z = off; off += up256(nwalk * 32 * sizeof(float));
  p.fast = d_k % grad::kTile == 0 && d_v % grad::kTile == 0;
  p.tc_ok = d_k % tcw::KT == 0 && d_v % tcw::VT == 0;
  p.Lp = p.C * tcw::CH;
  if (p.fast) {
    // fp32 qb / kf [BH][L][d_k], or their bf16 hi / lo parts [BH][Lp][d_k]
    const size_t nop = BH * static_cast<size_t>(p.tc_ok ? p.Lp : L) * d_k * sizeof(float);
    p.off_qb = off; off += up256(nop);
    p.off_kf = off; off += up256(nop);
  }
  p.bytes = off;
  return p;
}

template <typename Tin, typename Tout, typename Tg>
void launch_param_rows(const grad::ParamArgs& a, unsigned grid, bool vec, cudaStream_t st) {
  if (vec) grad::param_rows_kernel<Tin, Tout, Tg, true><<<grid, 256, 0, st>>>(a);
  else grad::param_rows_kernel<Tin, Tout, Tg, false><<<grid, 256, 0, st>>>(a);
}

template <typename Tin, typename Tout>
void launch_param_rows_g(const grad::ParamArgs& a, unsigned grid, bool vec, ret_dtype g_dt,
                         cudaStream_t st) {
  if (g_dt == RET_F32) launch_param_rows<Tin, Tout, float>(a, grid, vec, st);
  else launch_param_rows<Tin, Tout, __nv_bfloat16>(a, grid, vec, st);
}

template <typename Tx, typename Tg, int NV>
void launch_gn_backward_nv(const void* x, const void* dy, const float* w, void* dx, float* wpart,
                           int H, int L, int d_v, int nseg, float eps, unsigned grid, bool vec,
                           cudaStream_t st) {
  const size_t smem = wpart ? static_cast<size_t>(8) * d_v * sizeof(float) : 0;
  if (vec) {   // rows staged through shared memory: [4 warps][2 stages][2 rows][x, dy][d_v]
    const size_t ssm = std::max(static_cast<size_t>(4 * 2 * 2 * 2) * d_v * sizeof(Tx), smem);
    auto kern = grad::gn_backward_async_kernel<Tx, Tg, NV>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ssm));
    kern<<<grid, 128, ssm, st>>>(static_cast<const Tx*>(x), static_cast<const Tx*>(dy), w,
                                 static_cast<Tg*>(dx), wpart, H, L, d_v, nseg, eps);
  } else {   // rows that are not whole 16-byte vectors
    grad::gn_backward_kernel<Tx, Tg, false, NV><<<grid, 128, smem, st>>>(
        static_cast<const Tx*>(x), static_cast<const Tx*>(dy), w, static_cast<Tg*>(dx), wpart, H,
        L, d_v, nseg, eps);
  }
}

// NV = channels per lane: the smallest of 8, 16, 32 with d_v ≤ 32·NV.
template <typename Tx, typename Tg>
void launch_gn_backward(const void* x, const void* dy, const float* w, void* dx, float* wpart,
                        int H, int L, int d_v, int nseg, float eps, unsigned grid, bool vec,
                        cudaStream_t st) {
  if (d_v <= 256)
    launch_gn_backward_nv<Tx, Tg, 8>(x, dy, w, dx, wpart, H, L, d_v, nseg, eps, grid, vec, st);
  else if (d_v <= 512)
    launch_gn_backward_nv<Tx, Tg, 16>(x, dy, w, dx, wpart, H, L, d_v, nseg, eps, grid, vec, st);
  else
    launch_gn_backward_nv<Tx, Tg, 32>(x, dy, w, dx, wpart, H, L, d_v, nseg, eps, grid, vec, st);
}

size_t gn_backward_bytes(int B, int H, int L, int d_v) {
  const size_t nseg = (static_cast<size_t>(L) + grad::kRowsPerBlock - 1) / grad::kRowsPerBlock;
  return up256(static_cast<size_t>(B) * H * nseg * 2 * d_v * sizeof(float));
}

bool ok_dt(ret_dtype d) { return d == RET_F32 || d == RET_BF16; }
}  // namespace

extern "C" {

ret_status ret_groupnorm(const void* x, ret_dtype x_dt, void* y, ret_dtype y_dt, int B, int H,
                         int L, int d_v, const ret_gn* gn, cudaStream_t stream) {
  Range nv("ret_groupnorm");
  if (!x || !y || !gn || !ok_dt(x_dt) || !ok_dt(y_dt) || !al16(x) || !al16(y)) return RET_EINVAL;
  if (B < 1 || H < 1 || L < 1 || d_v < 1 || d_v > 1024) return RET_EINVAL;
  const int64_t rows = static_cast<int64_t>(B) * H * L;
  if (rows >= (int64_t(1) << 31)) return RET_EINVAL;
  if (!(gn->eps > 0.f) || !std::isfinite(gn->eps)) return RET_EINVAL;
  if (x == y && x_dt != y_dt) return RET_EINVAL;   // in place only with one type
  if ((gn->weight && !al16(gn->weight)) || (gn->bias && !al16(gn->bias))) return RET_EINVAL;
  const size_t r = static_cast<size_t>(rows);
  if (x_dt == RET_F32 && y_dt == RET_F32)
    launch_groupnorm(static_cast<const float*>(x), static_cast<float*>(y), gn, H, L, d_v, r, stream);
  else if (x_dt == RET_F32)
    launch_groupnorm(static_cast<const float*>(x), static_cast<__nv_bfloat16*>(y), gn, H, L, d_v, r, stream);
  else if (y_dt == RET_F32)
    launch_groupnorm(static_cast<const __nv_bfloat16*>(x), static_cast<float*>(y), gn, H, L, d_v, r, stream);
  else
    launch_groupnorm(static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), gn, H, L, d_v, r,
                     stream);
  return last_launch();
}

ret_status ret_groupnorm_backward_plan(int B, int H, int L, int d_v, size_t* workspace_bytes) {
  if (!workspace_bytes || B < 1 || H < 1 || L < 1 || d_v < 1 || d_v > 1024) return RET_EINVAL;
  *workspace_bytes = gn_backward_bytes(B, H, L, d_v);
  return RET_OK;
}

ret_status ret_groupnorm_backward(const void* x, const void* d_y, ret_dtype x_dt,
                                  const float* weight, float eps, int B, int H, int L, int d_v,
                                  void* d_x, ret_dtype grad_dt, float* d_weight, float* d_bias,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Range nv("ret_groupnorm_backward");
  if (!x || !d_y || !d_x || !ok_dt(x_dt) || !ok_dt(grad_dt)) return RET_EINVAL;
  if (!al16(x) || !al16(d_y) || !al16(d_x) || (weight && !al16(weight))) return RET_EINVAL;
  if (B < 1 || H < 1 || L < 1 || d_v < 1 || d_v > 1024) return RET_EINVAL;
  if (static_cast<int64_t>(B) * H * L >= (int64_t(1) << 31)) return RET_EINVAL;
  if (!(eps > 0.f) || !std::isfinite(eps)) return RET_EINVAL;
  if (d_x == x || d_x == d_y) return RET_EINVAL;
  const int nseg = (L + grad::kRowsPerBlock - 1) / grad::kRowsPerBlock;
  const int64_t nblk = static_cast<int64_t>(B) * H * nseg;
  float* wpart = nullptr;
  if (d_weight || d_bias) {
    if (!workspace || !al16(workspace) || workspace_bytes < gn_backward_bytes(B, H, L, d_v))
      return RET_EWORKSPACE;
    wpart = static_cast<float*>(workspace);
  }
  const bool vec = d_v % 8 == 0;
  const unsigned grid = static_cast<unsigned>(nblk);
  {
    Mark m("gn_backward", stream);
    if (x_dt == RET_F32) {
      if (grad_dt == RET_F32)
        launch_gn_backward<float, float>(x, d_y, weight, d_x, wpart, H, L, d_v, nseg, eps, grid, vec, stream);
      else
        launch_gn_backward<float, __nv_bfloat16>(x, d_y, weight, d_x, wpart, H, L, d_v, nseg, eps, grid, vec, stream);
    } else {
      if (grad_dt == RET_F32)
        launch_gn_backward<__nv_bfloat16, float>(x, d_y, weight, d_x, wpart, H, L, d_v, nseg, eps, grid, vec, stream);
      else
        launch_gn_backward<__nv_bfloat16, __nv_bfloat16>(x, d_y, weight, d_x, wpart, H, L, d_v, nseg, eps, grid,
                                                         vec, stream);
    }
  }
  ret_status s = last_launch();
  if (s != RET_OK || !wpart) return s;
  Mark m("gn_param_finish", stream);
  grad::gn_param_finish_kernel<<<dim3((d_v + 31) / 32, H), 256, 0, stream>>>(wpart, d_weight, d_bias, B, H,
                                                                             d_v, nseg);
  return last_launch();
}

ret_status ret_chunkwise_param_grads_plan(int B, int H, int L, int d_k, int d_v,
                                          size_t* workspace_bytes) {
  if (!workspace_bytes || B < 1 || H < 1 || H > kMaxHeads || L < 1) return RET_EINVAL;
  if (d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) || d_v < 1 || d_v > 1024) return RET_EINVAL;
  *workspace_bytes = plan_param_grads(B, H, L, d_k, d_v).bytes;
  return RET_OK;
}

ret_status ret_chunkwise_param_grads(const void* q, const void* k, const void* v,
                                     const void* d_out, ret_dtype in_dt, const void* out,
                                     ret_dtype out_dt, const void* dq, const void* dk,
                                     const void* dv, ret_dtype grad_dt, const float* gamma,
                                     const float* theta, int B, int H, int L, int d_k, int d_v,
                                     int64_t pos0, const float* state_in,
                                     const float* d_state_out, float* d_gamma, float* d_theta,
                                     void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream) {
  Range nv("ret_chunkwise_param_grads");
  if (!ok_dt(in_dt) || !ok_dt(out_dt) || !ok_dt(grad_dt)) return RET_EINVAL;
  if (!d_gamma && !d_theta) return RET_EINVAL;
  if (B < 1 || H < 1 || H > kMaxHeads || L < 1) return RET_EINVAL;
  if (d_k < 2 || d_k > 2 * kMaxPairs || (d_k & 1) || d_v < 1 || d_v > 1024) return RET_EINVAL;
  if (pos0 < 0 || pos0 + L > kMaxPos) return RET_EINVAL;
  if (static_cast<int64_t>(B) * H * L >= (int64_t(1) << 31)) return RET_EINVAL;
  for (const void* ptr : {q, k, v, d_out})
    if (!ptr || !al16(ptr)) return RET_EINVAL;
  if (d_theta)
    for (const void* ptr : {dq, dk})
      if (!ptr || !al16(ptr)) return RET_EINVAL;
  if (d_gamma)
    for (const void* ptr : {out, dv})
      if (!ptr || !al16(ptr)) return RET_EINVAL;
  if (!gamma || !theta) return RET_EINVAL;
  CallConsts cc;
  ret_status s = make_consts(cc, gamma, theta, H, d_k, grad::kGradChunk, L);
  if (s != RET_OK) return s;
  for (int h = 0; h < H; ++h)
    if (!(gamma[h] > 0.f)) return RET_EINVAL;   // dγ divides by γ; the walks take log2 γ
  const ParamPlan p = plan_param_grads(B, H, L, d_k, d_v);
  const int64_t nwalk = static_cast<int64_t>(B) * H * p.ntk * p.ntv;
  if (static_cast<int64_t>(B) * H * p.nseg >= (int64_t(1) << 31) || nwalk >= (int64_t(1) << 31))
    return RET_EUNSUPPORTED;
  if (!workspace || !al16(workspace) || workspace_bytes < p.bytes) return RET_EWORKSPACE;
  char* ws = static_cast<char*>(workspace);
  // (1) row sums with the in-chunk weights
  grad::ParamArgs a{};
  a.q = q; a.k = k; a.v = v; a.d_out = d_out; a.out = out; a.dq = dq; a.dk = dk; a.dv = dv;
  a.H = H; a.L = L; a.d_k = d_k; a.d_v = d_v; a.nseg = p.nseg;
  a.gpart = d_gamma ? reinterpret_cast<double*>(ws + p.off_g) : nullptr;
  a.tpart = d_theta ? reinterpret_cast<float*>(ws + p.off_t) : nullptr;
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(B) * H * p.nseg);
  const bool vec = d_k % 8 == 0 && d_v % 8 == 0;
  {
    Mark m("param_rows", stream);
    if (in_dt == RET_F32) {
      if (out_dt == RET_F32) launch_param_rows_g<float, float>(a, grid, vec, grad_dt, stream);
      else launch_param_rows_g<float, __nv_bfloat16>(a, grid, vec, grad_dt, stream);
    } else {
      if (out_dt == RET_F32) launch_param_rows_g<__nv_bfloat16, float>(a, grid, vec, grad_dt, stream);
      else launch_param_rows_g<__nv_bfloat16, __nv_bfloat16>(a, grid, vec, grad_dt, stream);
    }
  }
  if ((s = last_launch()) != RET_OK) return s;
  // (2) the state walks in fp32 and their boundary products
  float2* cs = reinterpret_cast<float2*>(ws + p.off_cs);
  {
    Mark m("param_angles", stream);
    const size_t n = static_cast<size_t>(L) * (d_k / 2);
    tcc::angle_table_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
        cs, cc, L, d_k / 2, static_cast<float>(pos0));
  }
  grad::WalkArgs w{};
  w.states = reinterpret_cast<float*>(ws + p.off_states);
  w.cs = cs;
  w.gpart = reinterpret_cast<double*>(ws + p.off_gw);
  w.zpart = reinterpret_cast<float*>(ws + p.off_z);
  w.H = H; w.L = L; w.d_k = d_k; w.d_v = d_v; w.C = p.C; w.ntk = p.ntk; w.ntv = p.ntv;
  w.pos0 = static_cast<float>(pos0);
  w.cc = cc;
  grad::WalkArgs fw = w;
  fw.a = k; fw.b = v; fw.s0 = state_in; fw.s_in = nullptr;
  fw.ascale = cc.kscale;
  grad::WalkArgs bw = w;
  bw.a = q; bw.b = d_out; bw.s0 = d_state_out; bw.s_in = state_in;
  bw.ascale = 1.f;
  const int64_t BH64 = static_cast<int64_t>(B) * H;
  if (p.tc_ok && in_dt == RET_BF16 && g_force_path != RET_PATH_SIMT && BH64 <= 65535) {
    // tensor-core walks on hi + lo bf16 operands
    const size_t half = static_cast<size_t>(BH64) * p.Lp * d_k;
    auto* qh = reinterpret_cast<__nv_bfloat16*>(ws + p.off_qb);
    auto* kh = reinterpret_cast<__nv_bfloat16*>(ws + p.off_kf);
    __nv_bfloat16* ql = qh + half;
    __nv_bfloat16* kl = kh + half;
    const size_t rows = static_cast<size_t>(BH64) * p.Lp;
    const size_t n = rows * (d_k / 8);
    {
      Mark m("param_prep", stream);
      tcw::walk_prep_tc_kernel<__nv_bfloat16><<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), qh, ql, kh, kl, cs, cc, H,
          L, p.Lp, d_k, rows);
    }
    CUtensorMap mv, mdo, mkh, mkl, mqh, mql;
    if (!make_map3(&mv, v, static_cast<uint64_t>(BH64), static_cast<uint64_t>(L), d_v) ||
        !make_map3(&mdo, d_out, static_cast<uint64_t>(BH64), static_cast<uint64_t>(L), d_v) ||
        !make_map(&mkh, kh, rows, d_k) || !make_map(&mkl, kl, rows, d_k) ||
        !make_map(&mqh, qh, rows, d_k) || !make_map(&mql, ql, rows, d_k))
      return RET_ECUDA;
    tcw::WalkTcArgs t{};
    t.states = w.states;
    t.gpart = w.gpart;
    t.zpart = w.zpart;
    t.H = H; t.L = L; t.Lp = p.Lp; t.d_k = d_k; t.d_v = d_v; t.C = p.C;
    t.pos0 = static_cast<float>(pos0);
    tcw::WalkTcArgs tf = t, tb = t;
    tf.s0 = state_in;
    tb.s0 = d_state_out;
    tb.s_in = state_in;
    const dim3 grid(static_cast<unsigned>(d_v / tcw::VT), static_cast<unsigned>(d_k / tcw::KT),
                    static_cast<unsigned>(BH64));
    auto walk = [&](auto kern, const CUtensorMap& mb, const CUtensorMap& mh, const CUtensorMap& ml,
                    const tcw::WalkTcArgs& wa, const char* name) {
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(tcw::SMEM_BYTES));
      Mark m(name, stream);
      kern<<<grid, tcw::NTHREADS, tcw::SMEM_BYTES, stream>>>(mb, mh, ml, wa, cc);
    };
    walk(tcw::walk_tc_kernel<true>, mv, mkh, mkl, tf, "param_walk_fwd");
    walk(tcw::walk_tc_kernel<false>, mdo, mqh, mql, tb, "param_walk_bwd");
    if ((s = last_launch()) != RET_OK) return s;
  } else if (p.fast) {
    float* qb = reinterpret_cast<float*>(ws + p.off_qb);
    float* kf = reinterpret_cast<float*>(ws + p.off_kf);
    const size_t rows = static_cast<size_t>(B) * H * L;
    const size_t n = rows * (d_k / 8);
    {
      Mark m("param_prep", stream);
      if (in_dt == RET_F32)
        grad::walk_prep_kernel<float><<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k), qb, kf, cs, cc, H, L, d_k, rows);
      else
        grad::walk_prep_kernel<__nv_bfloat16><<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), qb, kf, cs, cc, H, L,
            d_k, rows);
    }
    auto walk = [&](auto kern, const grad::WalkArgs& wa, const float* aop, int smem, const char* name) {
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      Mark m(name, stream);
      kern<<<static_cast<unsigned>(nwalk), 64, smem, stream>>>(wa, aop);
    };
    if (in_dt == RET_F32) {
      walk(grad::state_walk2_kernel<float, true>, fw, kf, grad::Walk2Smem<float>::BYTES, "param_walk_fwd");
      walk(grad::state_walk2_kernel<float, false>, bw, qb, grad::Walk2Smem<float>::BYTES, "param_walk_bwd");
    } else {
      walk(grad::state_walk2_kernel<__nv_bfloat16, true>, fw, kf, grad::Walk2Smem<__nv_bfloat16>::BYTES,
           "param_walk_fwd");
      walk(grad::state_walk2_kernel<__nv_bfloat16, false>, bw, qb, grad::Walk2Smem<__nv_bfloat16>::BYTES,
           "param_walk_bwd");
    }
    if ((s = last_launch()) != RET_OK) return s;
  } else {
    {
      Mark m("param_walk_fwd", stream);
      if (in_dt == RET_F32) grad::state_walk_fwd_kernel<float><<<static_cast<unsigned>(nwalk), 256, 0, stream>>>(fw);
      else grad::state_walk_fwd_kernel<__nv_bfloat16><<<static_cast<unsigned>(nwalk), 256, 0, stream>>>(fw);
    }
    if ((s = last_launch()) != RET_OK) return s;
    {
      Mark m("param_walk_bwd", stream);
      if (in_dt == RET_F32) grad::state_walk_bwd_kernel<float><<<static_cast<unsigned>(nwalk), 256, 0, stream>>>(bw);
      else grad::state_walk_bwd_kernel<__nv_bfloat16><<<static_cast<unsigned>(nwalk), 256, 0, stream>>>(bw);
    }
    if ((s = last_launch()) != RET_OK) return s;
  }
  // (3) fixed-order finishing sums
  grad::FinishArgs f{};
  f.gpart = a.gpart; f.gwalk = w.gpart; f.tpart = a.tpart; f.zpart = w.zpart;
  f.d_gamma = d_gamma; f.d_theta = d_theta;
  f.B = B; f.H = H; f.nseg = p.nseg; f.P = d_k / 2; f.ntk = p.ntk; f.ntv = p.ntv;
  for (int h = 0; h < H; ++h) f.inv_gamma[h] = 1.0 / static_cast<double>(gamma[h]);
  Mark m("param_finish", stream);
  grad::param_finish_kernel<<<static_cast<unsigned>(H + d_k / 2), 256, 0, stream>>>(f);
  return last_launch();
}

ret_status ret_sync_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return RET_ECUDA;
  unsigned int h[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(h, g_ret_status, sizeof(h)) != cudaSuccess) return RET_ECUDA;
  if (h[0] != 0u) {
    const unsigned int z[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_ret_status, z, sizeof(z)) != cudaSuccess) return RET_ECUDA;
    if (h[0] & kStatusTimeout) return RET_ETIMEOUT;
  }
  return RET_OK;
}

ret_status ret_selftest_timeout(int budget_us, cudaStream_t stream) {
  if (budget_us < 1 || budget_us > 2000000) return RET_EINVAL;
  int dev = 0, khz = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RET_ECUDA;
  if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess) return RET_ECUDA;
  if (khz <= 0) khz = 2000000;
  const long long cycles = static_cast<long long>(budget_us) * (khz / 1000);
  simt::selftest_timeout_kernel<<<1, 32, 0, stream>>>(cycles);
  return last_launch();
}

}  // extern "C"
