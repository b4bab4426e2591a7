// Chunkwise retention on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Form («从RoPE到Retention…» §4.3; RetNet 保留网络 explainer 分块循环), per
// (b, h) with chunk b = 128, local indices j, m in the chunk, S the fp32 state
// entering the chunk, ζ_m = γ^{b−1−m}:
//   o_j = γ^{j+1} q′_j S + Σ_{m≤j} γ^{j−m} (q′_j·k′_m) v_m
//   S  ← fmaf(γ^b, S, ΔS),  ΔS = Σ_m (ζ_m k′_m)ᵀ v_m
// Rewriting with K̂′_m = ζ_m k′_m (ζ folded into the prologue),
// P̂ = Q′K̂′ᵀ masked to m ≤ j (plain causal mask, exact zeros), and
// Ŝ = bf16(γ^b S):
//   o_j = ω_j · (Q′Ŝ + P̂V)_j   with ω_j = γ^{j+1−b}
// because ω_j·γ^b = γ^{j+1} and ω_j·ζ_m = γ^{j−m}.  So one fp32 accumulator
// holds both output terms and the decay mask reduces to a per-row scale,
// which the front pass folds into row j of Q′ (it then reaches P̂ through
// Q′K̂′ᵀ), so the accumulator is stored as it is (γ^{b−1} ≥ 2^-60 keeps every
// factor in range; the host routes other heads to the fp32 path).
//
// Each CTA owns one (b·h, 128-wide d_v tile) and walks the chunks in order.
// Transposed products keep d_v on the 128 TMEM lanes:
//   P̂   [j × m]      = Q′ · K̂′ᵀ          A = Q′ (smem, K-major), B = K̂′ (K-major)
//   ΔSᵀ [v × k]      = Vᵀ · K̂′           A = Vᵀ (MN-major),      B = K̂′ (MN-major)
//   Õᵀ  [v × j]      = Ŝᵀ · Q′ᵀ          A = Ŝᵀ (TMEM, bf16),    B = Q′ (K-major)
//   Õᵀ  [v × j]     += Vᵀ · P̂ᵀ           A = Vᵀ (MN-major),      B = P̂ (K-major)
// issued in that order for every chunk.  TMEM columns: X = [0, 128) holds P̂
// and then, once P̂ has been read out, Õᵀ; D = [128, 128 + d_k) holds the
// whole ΔSᵀ; SH = [128 + d_k, 128 + 3d_k/2) holds Ŝᵀ in bf16 pairs.  The
// fp32 master state Sᵀ lives in the registers of the 16 drain warps (d_k/4
// values per thread).  Every drain releases its TMEM region as soon as its
// tcgen05.ld has completed, before the arithmetic and the stores, and ΔSᵀ
// takes one MMA per chunk, so K̂′ is free right after the second product
// and the next chunk's K̂′ load overlaps the last two products.
#pragma once

#include "common.cuh"
#include "tc_primitives.cuh"

namespace ret {
namespace tcc {

using namespace ret::tc;

constexpr int CH = 128;               // chunk length = tile rows
constexpr int VT = 128;               // d_v columns per CTA
constexpr int NCW = 16;               // drain ("compute") warps
constexpr int NWARPS = NCW + 2;       // + TMA producer + MMA issuer
constexpr int NTHREADS = NWARPS * 32;

enum Bar : int {
  Q_FULL = 0, K_FULL, V_FULL,         // TMA → MMA
  Q_EMPTY, K_EMPTY, V_EMPTY,          // MMA → TMA
  P_FULL,                             // QK done            (MMA → drain)
  X_READ,                             // P̂ read out of X     (drain → MMA)
  P_SMEM,                             // P̂ in shared memory  (drain → MMA)
  DS_FULL,                            // ΔS done            (MMA → drain)
  DS_FREE,                            // ΔS read out of D    (drain → MMA)
  SH_FREE,                            // QS done, Ŝ may be rewritten (MMA → drain)
  SH_READY,                           // Ŝ written          (drain → MMA)
  O_FULL,                             // PV done            (MMA → drain)
  X_FREE,                             // Õ read out of X     (drain → MMA)
  MMA_DONE, NBAR_
};

template <int DK>
struct Cfg {
  static_assert(DK == 64 || DK == 128 || DK == 256, "d_k");
  static constexpr int QBOX = DK / 64;            // 64-column boxes of Q′ / K̂′
  static constexpr int SPT = DK / 4;              // state values per drain thread
  static constexpr uint32_t BOX = CH * 64 * 2;    // 16 KB
  static constexpr uint32_t Q_BYTES = CH * DK * 2;
  static constexpr uint32_t V_BYTES = CH * VT * 2;
  static constexpr uint32_t P_BYTES = CH * CH * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + Q_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + V_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
  static constexpr uint32_t OFF_TPTR = OFF_BAR + NBAR_ * 8;
  static constexpr uint32_t USED = OFF_TPTR + 16;
  static constexpr uint32_t SMEM_BYTES = USED + 1024;   // slack for 1024-B alignment
  static constexpr uint32_t T_X = 0, T_D = 128, T_SH = 128 + DK;
  static constexpr uint32_t T_COLS = (128 + DK + DK / 2) <= 256 ? 256 : 512;
};

// Compile-time modes of the chunk kernels (template argument MODE, bits).
constexpr int kModeBwd = 1, kModeRev = 2, kModeFold = 4;

// Every field has a default (zero / null), so a ChunkArgs built field by
// field never carries garbage into a mode it does not set up.
struct ChunkArgs {
  const float* state_in = nullptr;   // per grid row [DK][d_v], or nullptr
  float* state_out = nullptr;        // or nullptr
  void* out = nullptr;               // [BH][seq_len][d_v] bf16, or fp32 when out_f32; nullptr: no output
  int out_f32 = 0;
  int H = 0, d_v = 0;
  int nchunks = 0;                   // chunks this CTA walks
  // One sequence: seq_len tokens (any length), seq_chunks chunks of 128,
  // seq_lp = 128·seq_chunks rows of it in the rotated Q′ / K̂′ workspace
  // (rows past seq_len are zero).  The last chunk has seq_len − 128·(seq_chunks−1)
  // tokens and carries with γ^that instead of γ^128.
  int seq_len = 0, seq_lp = 0, seq_chunks = 0;
  void* tail_out = nullptr;          // staging [sequences][128][d_v] (out's type) for a short
                                     // last chunk, or nullptr when seq_len is a multiple of 128
  // Chunk-parallel layout: the rows of grid.y are (sequence, chunk) pairs of
  // one chunk each: sequence = blockIdx.y / seq_div, chunk = blockIdx.y % seq_div,
  // head = sequence % H.  raw_ds: state_out receives the chunk's ΔS itself
  // instead of fmaf(γ^b, S, ΔS).
  int seq_div = 1, raw_ds = 0;
  // Grids with more rows than gridDim.y allows fold them over grid.z: row =
  // blockIdx.y + gridDim.y·blockIdx.z, and the CTAs past grid_rows exit at
  // once.  0: one row per blockIdx.y (gridDim.z = 1).  Only the
  // instantiations with kModeFold read it (the others take row = blockIdx.y).
  int grid_rows = 0;
  // V's sequence index is the row's sequence mod v_seqs (0: the sequence
  // itself), so that grid rows that differ only in a piece of the
  // contracted columns read one copy of V.
  int v_seqs = 0;
  // Gradient-pass instantiations only: the state is read as γ^s_in_exp ·
  // state_in and written as γ^s_out_exp · S (0: unscaled).
  int s_in_exp = 0, s_out_exp = 0;
  // Ring mode of the pair kernel (ring > 0, carried layout only): grid rows
  // [0, ring_prod_rows) are producer CTAs that rotate raw q, k (read through
  // their own tensor maps) into `ring` chunk slots per head — ring_q / ring_k
  // [ring_heads][ring][128][d_k] bf16 — and the rows after them are the
  // consumer pairs of heads ring_bh0 + (row − ring_prod_rows).  ring_flags
  // holds ready[ring] (producer CTAs done with a slot's chunk, cumulative) and
  // consumed[ring] (consumer pairs done loading it, cumulative); ring_cs is
  // the (cos, sin) table [seq_len][d_k/2]; ring_nbuf the producers' shared-
  // memory buffers.
  int ring = 0, ring_prod_rows = 0, ring_heads = 0, ring_bh0 = 0, ring_npairs = 0, ring_nbuf = 0;
  uint32_t* ring_flags = nullptr;
  __nv_bfloat16* ring_q = nullptr;
  __nv_bfloat16* ring_k = nullptr;
  const float2* ring_cs = nullptr;
};

// ---------------------------------------------------------------------------
// One 32-bit word (an interleaved pair x_{2i}, x_{2i+1} in bf16) rotated by
// the angle with cosine c and sine s and scaled by w, rounded to bf16:
//   Q″ pair: w·(a·c − b·s), w·(a·s + b·c)     (w = ω for Q″, 1 for Q′)
//   K̂′ pair: a·(zc) − b·(zs), a·(zs) + b·(zc) (z = d_k^{-1/2}·ζ, zc = z·c, zs = z·s)
// Every operation is rounded explicitly (no contraction left to the
// compiler), so the front pass and the ring producers of the chunk kernel
// produce the same bits from the same inputs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t rot_q_word(uint32_t w, float c, float s, float wq) {
  const float a = bf16lo_to_f32(w), b = bf16hi_to_f32(w);
  const float x = __fmaf_rn(a, c, __fmul_rn(-b, s));
  const float y = __fmaf_rn(a, s, __fmul_rn(b, c));
  return pack_bf16x2(__fmul_rn(wq, x), __fmul_rn(wq, y));
}
__device__ __forceinline__ uint32_t rot_k_word(uint32_t w, float zc, float zs) {
  const float a = bf16lo_to_f32(w), b = bf16hi_to_f32(w);
  return pack_bf16x2(__fmaf_rn(a, zc, __fmul_rn(-b, zs)), __fmaf_rn(a, zs, __fmul_rn(b, zc)));
}
// Per-row factors of the folded form for local position t of a sequence of
// L tokens (chunks of 128, the last one of length bc): ζ·d_k^{-1/2} for K̂′
// and ω for Q″ (1 when the ω fold is off).
__device__ __forceinline__ void row_factors(const CallConsts& cc, int h, int t, int L, int Lp, int chunk,
                                            int fold_omega, float& zk, float& wq) {
  const int bc = (t / chunk == Lp / chunk - 1) ? L - (Lp - chunk) : chunk;   // length of t's chunk
  const float e = static_cast<float>(bc - 1 - (t % chunk));
  const float ew = static_cast<float>((t % chunk) + 1 - bc);
  zk = __fmul_rn(cc.kscale, gpow(cc.lg2g[h], e));
  wq = fold_omega ? gpow(cc.lg2g[h], ew) : 1.f;
}

// ---------------------------------------------------------------------------
// (cos, sin) of the rotation angle (pos0 + t)·θ_i for t < L, i < d/2:
// cs[t][i], the table the ring producers read (one accurate sincos per
// (position, pair) for the whole call).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) angle_table_kernel(float2* __restrict__ cs, CallConsts cc,
                                                          int L, int half, float pos0) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(L) * half) return;
  const int t = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
  float c, s;
  angle_cs(pos0 + static_cast<float>(t), cc.theta[i], c, s);
  cs[idx] = make_float2(c, s);
}

// ---------------------------------------------------------------------------
// Front pass: Q′ = R(nθ)q and K̂′ = d_k^{-1/2}·ζ_{t mod b}·R(nθ)k in bf16.
// With fold_omega, Q′ row t also carries ω_{t mod b} = γ^{(t mod b)+1−b}:
// o_j = ω_j (Q′Ŝ + P̂V)_j, and scaling row j of Q′ scales both terms (P̂
// inherits it through Q′K̂′ᵀ), so the chunk kernels store their
// accumulator as it is.
// Thread ↔ (row t, 4 consecutive pairs); one sincos per pair shared by the
// heads of that row in the block's slice of heads (grid.y slices, one slice
// unless the rows alone give too few blocks), eight heads' loads in flight
// at a time; raw q and
// k are read with the evict-first hint.  q, k have L rows per head; Q′, K̂′
// have Lp = 128·⌈L/128⌉ rows per head, the rows past L written as zeros, and
// the last chunk's factors use its own length b_c (ζ = γ^{b_c−1−(t mod b)},
// ω = γ^{(t mod b)+1−b_c}).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rotate_qk_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    __nv_bfloat16* __restrict__ qo, __nv_bfloat16* __restrict__ ko, CallConsts cc, int BH,
    int H, int L, int Lp, int d, float pos0, int chunk, int fold_omega, RowPos rp) {
  constexpr int U = 8;   // heads in flight per thread (the pass is HBM-bound)
  const int vecs = d / 8;
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(Lp) * vecs) return;
  // Positions are walked last to first, so the first chunks the main kernel
  // reads are the last ones written and are still in L2.
  const int tt = static_cast<int>(idx / vecs), cidx = static_cast<int>(idx % vecs);
  const int t = Lp - 1 - tt;
  const size_t ostride = static_cast<size_t>(Lp) * d;   // output elements between heads
  const size_t oofs = static_cast<size_t>(t) * d + 8 * cidx;
  // grid.y splits the heads into slices (short sequences: enough blocks)
  const int hpy = (BH + static_cast<int>(gridDim.y) - 1) / static_cast<int>(gridDim.y);
  const int y0 = static_cast<int>(blockIdx.y) * hpy, y1 = min(BH, y0 + hpy);
  if (t >= L) {   // padding rows of the last chunk
    for (int bh = y0; bh < y1; ++bh) {
      *reinterpret_cast<uint4*>(qo + oofs + static_cast<size_t>(bh) * ostride) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(ko + oofs + static_cast<size_t>(bh) * ostride) = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  const size_t hstride = static_cast<size_t>(L) * d;   // input elements between heads
  const size_t off0 = static_cast<size_t>(t) * d + 8 * cidx;
  // Heads [bh_lo, bh_hi) whose rows start at position `start`.
  auto rows = [&](float start, int bh_lo, int bh_hi) {
    float c[4], s[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) angle_cs(start + static_cast<float>(t), cc.theta[4 * cidx + u], c[u], s[u]);
    for (int bh0 = bh_lo; bh0 < bh_hi; bh0 += U) {
      uint4 qv[U], kv[U];
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        if (bh0 + uu < bh_hi) {
          const size_t off = off0 + static_cast<size_t>(bh0 + uu) * hstride;
          qv[uu] = __ldcs(reinterpret_cast<const uint4*>(q + off));
          kv[uu] = __ldcs(reinterpret_cast<const uint4*>(k + off));
        }
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const int bh = bh0 + uu;
        if (bh >= bh_hi) break;
        float zk, wq;
        row_factors(cc, bh % H, t, L, Lp, chunk, fold_omega, zk, wq);
        const uint32_t qw[4] = {qv[uu].x, qv[uu].y, qv[uu].z, qv[uu].w};
        const uint32_t kw[4] = {kv[uu].x, kv[uu].y, kv[uu].z, kv[uu].w};
        uint32_t qr[4], kr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          qr[u] = rot_q_word(qw[u], c[u], s[u], wq);
          kr[u] = rot_k_word(kw[u], __fmul_rn(zk, c[u]), __fmul_rn(zk, s[u]));
        }
        const size_t off = oofs + static_cast<size_t>(bh) * ostride;
        *reinterpret_cast<uint4*>(qo + off) = make_uint4(qr[0], qr[1], qr[2], qr[3]);
        *reinterpret_cast<uint4*>(ko + off) = make_uint4(kr[0], kr[1], kr[2], kr[3]);
      }
    }
  };
  if (!rp.on) {
    rows(pos0, y0, y1);   // one sincos per (position, pair) for the slice's heads
  } else {
    for (int b = y0 / H; b * H < y1; ++b) rows(rp.p[b], max(b * H, y0), min(b * H + H, y1));
  }
}

// ---------------------------------------------------------------------------
// Rows 0 … T−1 of each sequence's staged last chunk ([BH][128][row_vecs]
// 16-byte vectors) to rows row0 … row0+T−1 of out ([BH][L][row_vecs]).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) tail_copy_kernel(const uint4* __restrict__ src,
                                                        uint4* __restrict__ dst, int BH, int T,
                                                        int L, int row0, int row_vecs) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t per = static_cast<size_t>(T) * row_vecs;
  if (idx >= per * BH) return;
  const size_t bh = idx / per, rem = idx % per;
  const size_t r = rem / row_vecs, c = rem % row_vecs;
  dst[(bh * L + row0 + r) * row_vecs + c] = src[(bh * CH + r) * row_vecs + c];
}

// ---------------------------------------------------------------------------
// Main kernel.  grid = (⌈d_v / 128⌉, B·H); block = 576 threads; 1 CTA per SM.
// Warp 0: TMA producer.  Warp 1: MMA issuer.  Warps 2..17: drain warps; the
// drain warp with hardware warp id w reads TMEM lanes 32·(w % 4) … +31
// (v for Õᵀ/ΔSᵀ/Ŝᵀ, j for P̂) and handles column slice (w − 2) / 4.
// MODE: bits kModeBwd (the gradient pass's instantiations, carried layout:
// V's sequence index taken mod args.v_seqs, the state scaled on entry and
// exit), kModeRev (the anti-causal form: chunks walked from the last to the
// first, key m kept for query j when m ≥ j) and kModeFold (grid rows folded
// over grid.z).  The plain forward instantiation (MODE = 0) compiles none
// of it, so its rows are blockIdx.y itself.
// ---------------------------------------------------------------------------
template <int DK, int MODE = 0>
__global__ void __launch_bounds__(NTHREADS, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, ChunkArgs args, CallConsts cc) {
  using C = Cfg<DK>;
  constexpr bool BWD = (MODE & kModeBwd) != 0, REV = (MODE & kModeRev) != 0,
                 FOLD = (MODE & kModeFold) != 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + C::OFF_Q, sK = sb + C::OFF_K, sV = sb + C::OFF_V, sP = sb + C::OFF_P;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v0 = blockIdx.x * VT;
  const int bh = FOLD ? static_cast<int>(blockIdx.y + gridDim.y * blockIdx.z) : static_cast<int>(blockIdx.y);
  if (FOLD && args.grid_rows && bh >= args.grid_rows) return;   // past the rows of a folded grid
  const int seq = bh / args.seq_div, c0 = bh % args.seq_div;   // sequence; its first chunk here
  const int h = seq % args.H;
  const int d_v = args.d_v, nch = args.nchunks;
  // γ^{b_c} of chunk c of the sequence (its last chunk may be shorter)
  auto gch = [&](int c) -> float { return c == args.seq_chunks - 1 ? cc.gtail[h] : cc.gb[h]; };
  // chunk of the sequence handled at step i
  auto cix = [&](int i) -> int { return REV ? nch - 1 - i : c0 + i; };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int i = 0; i < NBAR_; ++i) {
      const bool from_drain = (i == X_READ || i == P_SMEM || i == DS_FREE || i == SH_READY ||
                               i == X_FREE);
      mbar_init(bar(i), from_drain ? NCW : 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + C::OFF_TPTR, C::T_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_TPTR);

  if (warp == 0) {
    // ------------------------------ TMA producer ---------------------------
    // Buffers free up in the order K̂′ (after ΔS), Q′ (after QS), V (after PV).
    if (lane == 0) {
      int issued = -1;   // last chunk whose loads were all issued
      const int vseq = BWD && args.v_seqs ? seq % args.v_seqs : seq;   // V's row in its tensor map
      for (int i = 0; i < nch; ++i) {
        const uint32_t pp = static_cast<uint32_t>(i - 1) & 1u;
        const int y = seq * args.seq_lp + cix(i) * CH;   // row of Q′ / K̂′
        const int yv = cix(i) * CH;                       // row of V within the sequence
        if (i > 0 && !mbar_wait(bar(K_EMPTY), pp, 0x101)) break;
        mbar_arrive_expect_tx(bar(K_FULL), C::Q_BYTES);
        for (int b = 0; b < C::QBOX; ++b) tma_load_2d(sK + b * C::BOX, &tm_k, 64 * b, y, bar(K_FULL));
        if (i > 0 && !mbar_wait(bar(Q_EMPTY), pp, 0x102)) break;
        mbar_arrive_expect_tx(bar(Q_FULL), C::Q_BYTES);
        for (int b = 0; b < C::QBOX; ++b) tma_load_2d(sQ + b * C::BOX, &tm_q, 64 * b, y, bar(Q_FULL));
        if (i > 0 && !mbar_wait(bar(V_EMPTY), pp, 0x103)) break;
        mbar_arrive_expect_tx(bar(V_FULL), C::V_BYTES);
        for (int b = 0; b < 2; ++b) tma_load_3d(sV + b * C::BOX, &tm_v, v0 + 64 * b, yv, vseq, bar(V_FULL));
        issued = i;
      }
      if (issued >= 0 && status_aborted()) {
        const uint32_t pl = static_cast<uint32_t>(issued) & 1u;
        mbar_wait(bar(K_FULL), pl, 0x1f1, kWaitBudgetCycles / 8);
        mbar_wait(bar(Q_FULL), pl, 0x1f2, kWaitBudgetCycles / 8);
        mbar_wait(bar(V_FULL), pl, 0x1f3, kWaitBudgetCycles / 8);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer -----------------------------
    if (lane == 0) {
      const uint32_t tX = tmem + C::T_X, tD = tmem + C::T_D, tSH = tmem + C::T_SH;
      constexpr uint32_t ID_P = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t ID_QS = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t ID_PV = idesc_bf16_f32(128, 128, 1, 0);
      constexpr uint32_t ID_KV = idesc_bf16_f32(128, DK, 1, 1);
      // Shared-memory descriptors are built once; every k-step adds its byte
      // offset / 16 to the start-address field (no carry: all operands sit
      // below 256 KB), so the unrolled issue loops cost a few integer adds
      // per MMA and the single issuing thread keeps ahead of the tensor core.
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);      // K-major Q′
      const uint64_t dK = sdesc_sw128(sK, 16, 1024);      // K-major K̂′
      const uint64_t dKm = sdesc_sw128(sK, C::BOX, 1024); // MN-major K̂′
      const uint64_t dV = sdesc_sw128(sV, C::BOX, 1024);  // MN-major V
      const uint64_t dP = sdesc_sw128(sP, 16, 1024);      // K-major P̂
      auto kmaj = [](int s) -> uint64_t {                 // k-step s of a K-major tile
        return static_cast<uint64_t>(((s >> 2) * C::BOX + (s & 3) * 32) >> 4);
      };
      for (int i = 0; i < nch; ++i) {
        const uint32_t pi = static_cast<uint32_t>(i) & 1u;
        const uint32_t pp = static_cast<uint32_t>(i - 1) & 1u;
        // 1. P̂ = Q′ K̂′ᵀ into X (needs Õ of the previous chunk read out)
        if (!mbar_wait(bar(K_FULL), pi, 0x201)) break;
        if (!mbar_wait(bar(Q_FULL), pi, 0x202)) break;
        if (i > 0 && !mbar_wait(bar(X_FREE), pp, 0x203)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < DK / 16; ++s) mma_ss(tX, dQ + kmaj(s), dK + kmaj(s), ID_P, s > 0 ? 1u : 0u);
        mma_commit(bar(P_FULL));
        // 2. ΔSᵀ = Vᵀ K̂′ into D (needs the previous ΔS read out)
        if (!mbar_wait(bar(V_FULL), pi, 0x204)) break;
        if (i > 0 && !mbar_wait(bar(DS_FREE), pp, 0x205)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < CH / 16; ++s)
          mma_ss(tD, dV + static_cast<uint64_t>(s * 128), dKm + static_cast<uint64_t>(s * 128), ID_KV,
                 s > 0 ? 1u : 0u);   // +2048 bytes (16 rows) per step
        mma_commit(bar(DS_FULL));
        mma_commit(bar(K_EMPTY));
        // 3. Õᵀ = Ŝᵀ Q′ᵀ into X (needs P̂ read out and Ŝ of the previous chunk)
        if (!mbar_wait(bar(X_READ), pi, 0x206)) break;
        if (!mbar_wait(bar(SH_READY), pi, 0x207)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < DK / 16; ++s) mma_ts(tX, tSH + s * 8, dQ + kmaj(s), ID_QS, s > 0 ? 1u : 0u);
        mma_commit(bar(Q_EMPTY));
        mma_commit(bar(SH_FREE));
        // 4. Õᵀ += Vᵀ P̂ᵀ (needs the masked bf16 P̂ in shared memory)
        if (!mbar_wait(bar(P_SMEM), pi, 0x208)) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < CH / 16; ++s)
          mma_ss(tX, dV + static_cast<uint64_t>(s * 128), dP + kmaj(s), ID_PV, 1u);
        mma_commit(bar(O_FULL));
        mma_commit(bar(V_EMPTY));
      }
      // All issued MMAs must finish before TMEM is released.
      mma_commit(bar(MMA_DONE));
      mbar_wait(bar(MMA_DONE), 0, 0x2ff);
    }
  } else {
    // ------------------------------ drain warps ----------------------------
    const int w = warp - 2;                 // 0..15
    const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
    const int cs = w >> 2;                  // 32-column slice for P̂ / Õ drains
    const int kr = w >> 2;                  // state k range [kr*SPT, kr*SPT+SPT)
    const int vl = 32 * quarter + lane;     // local v (TMEM lane) for Õ / ΔS / Ŝ
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    const size_t sbase = static_cast<size_t>(bh) * DK * d_v + v0 + vl;
    // A tile narrower than 128 (d_v = 64): lanes past d_v only carry zeros
    // (V's missing columns read as zeros) and touch no memory.
    const bool vlive = v0 + vl < d_v;

    float S[C::SPT];
#pragma unroll
    for (int u = 0; u < C::SPT; ++u)
      S[u] = (args.state_in && vlive) ? args.state_in[sbase + static_cast<size_t>(kr * C::SPT + u) * d_v] : 0.f;
    if constexpr (BWD) {
      if (args.s_in_exp) {
        const float f = gpow(cc.lg2g[h], static_cast<float>(args.s_in_exp));
#pragma unroll
        for (int u = 0; u < C::SPT; ++u) S[u] *= f;
      }
    }

    // Ŝᵀ = bf16(γ^b S) for this thread's v lane and k range.
    auto write_shat = [&](float g) {
#pragma unroll
      for (int c = 0; c < C::SPT / 16; ++c) {
        uint32_t pk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          pk[u] = pack_bf16x2(g * S[c * 16 + 2 * u], g * S[c * 16 + 2 * u + 1]);
        tmem_st8(tmem + C::T_SH + lane_off + (kr * C::SPT + c * 16) / 2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(SH_READY));
    };
    write_shat(gch(cix(0)));

    bool ok = true;
    for (int i = 0; i < nch && ok; ++i) {
      const uint32_t pi = static_cast<uint32_t>(i) & 1u;
      const float gi = gch(cix(i));
      // ---- (a) P̂ drain: causal mask, bf16, into the K-major swizzled tile ----
      if (!mbar_wait(bar(P_FULL), pi, 0x301)) { ok = false; break; }
      tc_fence_after();
      {
        // Two rounds of two 8-column loads per wait keep the register peak low
        // (S stays live) while halving the TMEM round trips; X is released
        // after the last load.
        const int j = vl;   // row of P̂ = TMEM lane
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t r[16];
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&r[0]));
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 16 * hf + 8, *reinterpret_cast<uint32_t(*)[8]>(&r[8]));
          tmem_ld_wait();
          if (hf == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(X_READ));
          }
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t pk[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int m = 32 * cs + 16 * hf + 8 * g + 2 * u;
              const bool ka = REV ? m >= j : m <= j, kb = REV ? m + 1 >= j : m + 1 <= j;
              const float a = ka ? __uint_as_float(r[8 * g + 2 * u]) : 0.f;
              const float b = kb ? __uint_as_float(r[8 * g + 2 * u + 1]) : 0.f;
              pk[u] = pack_bf16x2(a, b);
            }
            const int m0 = 32 * cs + 16 * hf + 8 * g;
            st_shared_v4(sP + (m0 >> 6) * C::BOX + sw128_offset(j, m0 & 63), pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(P_SMEM));

      // ---- (b) ΔS drain: S = fmaf(γ^b, S, ΔS) ----
      if (!mbar_wait(bar(DS_FULL), pi, 0x302)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < C::SPT / 16; ++c) {
        uint32_t d[16];
        tmem_ld16(tmem + C::T_D + lane_off + kr * C::SPT + c * 16, d);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; ++u)
          S[16 * c + u] = args.raw_ds ? __uint_as_float(d[u]) : fmaf(gi, S[16 * c + u], __uint_as_float(d[u]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(DS_FREE));

      // ---- (c) Ŝ for the next chunk, once QS of this chunk has read Ŝ ----
      if (!mbar_wait(bar(SH_FREE), pi, 0x303)) { ok = false; break; }
      tc_fence_after();
      write_shat(gch(cix(i + 1)));

      // ---- (d) Õ drain: release X, then store (ω_j rides on Q′) ----
      if (!mbar_wait(bar(O_FULL), pi, 0x304)) { ok = false; break; }
      tc_fence_after();
      {
        // A short last chunk goes whole to the staging tile [sequence][128][d_v]
        // (a copy kernel then moves its valid rows), so no store needs a check.
        const bool staged = args.tail_out && cix(i) == args.seq_chunks - 1;
        void* const obuf = staged ? args.tail_out : args.out;
        const size_t base = staged
            ? (static_cast<size_t>(seq) * CH + 32 * cs) * d_v + v0 + vl
            : (static_cast<size_t>(seq) * args.seq_len + static_cast<size_t>(cix(i)) * CH + 32 * cs) * d_v + v0 + vl;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t r[16];
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&r[0]));
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 16 * hf + 8, *reinterpret_cast<uint32_t(*)[8]>(&r[8]));
          tmem_ld_wait();
          if (hf == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(X_FREE));
          }
          const size_t gb0 = base + static_cast<size_t>(16 * hf) * d_v;
          if (!args.out || !vlive) {
          } else if (args.out_f32) {
            float* o = reinterpret_cast<float*>(obuf) + gb0;
#pragma unroll
            for (int c = 0; c < 16; ++c) o[static_cast<size_t>(c) * d_v] = __uint_as_float(r[c]);
          } else {
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(obuf) + gb0;
#pragma unroll
            for (int c = 0; c < 16; ++c) o[static_cast<size_t>(c) * d_v] = __float2bfloat16_rn(__uint_as_float(r[c]));
          }
        }
      }
    }
    if (ok && args.state_out && vlive) {
#pragma unroll
      for (int u = 0; u < C::SPT; ++u)
        args.state_out[sbase + static_cast<size_t>(kr * C::SPT + u) * d_v] =
            BWD && args.s_out_exp ? S[u] * gpow(cc.lg2g[h], static_cast<float>(args.s_out_exp)) : S[u];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::T_COLS);
  }
}

}  // namespace tcc
}  // namespace ret
