// Chunkwise retention on a CTA pair (tcgen05 cta_group::2).
//
// Same arithmetic as the single-CTA chunk kernel (kernel_tc_chunk.cuh: form
// of «从RoPE到Retention…» §4.3 and the RetNet 保留网络 explainer 分块循环,
// rewritten with K̂′_m = ζ_m k′_m, P̂ = causal(Q′K̂′ᵀ), Ŝ = bf16(γ^b S),
// o_j = ω_j (Q′Ŝ + P̂V)_j, S ← fmaf(γ^b, S, ΔS)), but the two CTAs that own
// the d_v tiles 2p and 2p+1 of one (b, h) form a cluster and run every
// product as one pair MMA issued by the even CTA:
//   P̂   [j × m]  = Q′ · K̂′ᵀ     M = 128: each CTA holds its 64 query rows of
//                                Q′ and one half of the keys of K̂′
//   ΔSᵀ [v × k]  = Vᵀ · K̂′      M = 256: each CTA its own V tile and one
//                                half of the d_k columns of K̂′
//   Õᵀ  [v × j]  = Ŝᵀ · Q′ᵀ     M = 256: Ŝᵀ from each CTA's TMEM, Q′ rows
//                                split by query half
//   Õᵀ  [v × j] += Vᵀ · P̂ᵀ      M = 256: P̂ rows split by query half
// So each CTA stages half of Q′ and half of P̂ instead of all of them, and
// the operand reads from shared memory per CTA drop by about 40%, which
// leaves room to double-buffer Q′ and V.  The query half of P̂ each CTA
// drains is exactly the half its own PV operand needs, so no P̂ crosses
// between the CTAs; each CTA still drains its own Õᵀ, ΔSᵀ and keeps its
// own fp32 state tile, as in the single-CTA kernel, and the results are
// the same numbers in the same order.
//
// Per chunk the products are issued ΔS, QK, QS, PV.  The chain that bounds
// a chunk is QK → P̂ drain → QS → PV → Õ drain → next QK (P̂ and Õᵀ share
// TMEM columns), and ΔS of the next chunk, which needs neither, runs on
// the tensor cores while the drains store Õ.  K̂′ is staged as two pieces
// with their own barriers (the key half with all d_k for QK, all keys with
// a d_k half for ΔS), each reloaded as soon as its product is done.
//
// Synchronisation: TMA loads of both CTAs count their bytes on the even
// CTA's FULL barriers; pair commits arrive on the barriers of both CTAs;
// drain warps of both CTAs arrive on the even CTA's barriers (CTA-scope
// release after their TMEM / shared-memory hand-off has completed).
#pragma once

#include "common.cuh"
#include "tc_primitives.cuh"
#include "kernel_tc_chunk.cuh"

namespace ret {
namespace tcq {

using namespace ret::tc;
using tcc::ChunkArgs;
using tcc::CH;
using tcc::NCW;
using tcc::NTHREADS;
using tcc::VT;
using tcc::rot_k_word;
using tcc::rot_q_word;
using tcc::row_factors;

enum Bar : int {
  // TMA → MMA (the even CTA's copy counts both CTAs' bytes)
  Q_FULL0 = 0, Q_FULL1, V_FULL0, V_FULL1, KQ_FULL, KV_FULL,
  // MMA → TMA (both CTAs)
  Q_EMPTY0, Q_EMPTY1, V_EMPTY0, V_EMPTY1, KQ_EMPTY, KV_EMPTY,
  P_FULL,     // QK done                      (MMA → drains)
  X_READ,     // P̂ read out of X              (drains → MMA)
  P_SMEM,     // P̂ halves in shared memory    (drains → MMA)
  DS_FULL,    // ΔS done                      (MMA → drains)
  DS_FREE,    // ΔS read out of D             (drains → MMA)
  SH_FREE,    // QS done, Ŝ may be rewritten  (MMA → drains)
  SH_READY,   // Ŝ written                    (drains → MMA)
  O_FULL,     // PV done                      (MMA → drains)
  X_FREE,     // Õ read out of X              (drains → MMA)
  MMA_DONE, NBAR_
};

template <int DK>
struct Cfg {
  static_assert(DK == 128 || DK == 256, "d_k");
  static constexpr int QBOX = DK / 64;             // 64-column boxes across d_k
  static constexpr int SPT = DK / 4;               // state values per drain thread
  static constexpr uint32_t HBOX = 64 * 64 * 2;    // 64-row box, 8 KB
  static constexpr uint32_t BOX = CH * 64 * 2;     // 128-row box, 16 KB
  static constexpr uint32_t QH_BYTES = QBOX * HBOX;        // 64 query rows of Q′
  static constexpr uint32_t KQ_BYTES = QBOX * HBOX;        // 64 keys of K̂′, all d_k
  static constexpr uint32_t KV_BYTES = (QBOX / 2) * BOX;   // all keys, d_k / 2 columns
  static constexpr uint32_t V_BYTES = 2 * BOX;             // 128 keys × 128 v
  static constexpr uint32_t P_BYTES = 2 * HBOX;            // 64 query rows × 128 keys
  static constexpr uint32_t OFF_Q = 0;                     // two slots
  static constexpr uint32_t OFF_KQ = OFF_Q + 2 * QH_BYTES;
  static constexpr uint32_t OFF_KV = OFF_KQ + KQ_BYTES;
  static constexpr uint32_t OFF_V = OFF_KV + KV_BYTES;     // two slots
  static constexpr uint32_t OFF_P = OFF_V + 2 * V_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
  static constexpr uint32_t OFF_TPTR = OFF_BAR + NBAR_ * 8;
  static constexpr uint32_t USED = OFF_TPTR + 16;
  static constexpr uint32_t SMEM_BYTES = USED + 1024;     // slack for 1024-B alignment
  static constexpr uint32_t T_X = 0, T_D = 128, T_SH = 128 + DK;
  static constexpr uint32_t T_COLS = 512;
};

// ---------------------------------------------------------------------------
// Ring producer (ring mode, grid rows [0, ring_prod_rows); both CTAs of such
// a cluster are producers).  The P producer CTAs share the rows of every
// chunk: producer p rotates rows r ≡ p (mod P) of chunk c for all the
// launch's heads, chunk after chunk.  Per row, warp 16 loads the raw q and k
// rows of all heads (two 3-D TMA boxes of d_k × 1 × heads, streamed with an
// evict-first hint) and the row of the angle table into one of ring_nbuf
// shared-memory buffers; warps 0..15 rotate it (warp w takes heads w, w+16,
// …; each lane 8 consecutive columns) with the front pass's arithmetic
// (rot_q_word / rot_k_word / row_factors) into slot c mod R of the ring
// (angles from the call's table, or, when every batch row has its own start
// position, from angle_cs per head).
// Before its first row of chunk c a rotation warp waits until every
// consumer pair has loaded chunk c − R out of that slot; after its last row
// of chunk c the CTA publishes the slot (release) once all rotation warps
// are done.  Rows past the sequence's end are written as zeros.  After a
// failed wait a warp stops working but still reaches every named barrier.
// ---------------------------------------------------------------------------
template <int DK>
__device__ __forceinline__ void ring_producer(const CUtensorMap* tm_rq, const CUtensorMap* tm_rk,
                                              const ChunkArgs& a, const CallConsts& cc,
                                              const RowPos& rp, uint32_t sb) {
  constexpr int VECS = DK / 8;     // 16-byte vectors per row
  constexpr int HPW = 32 / VECS;   // heads per warp and round
  constexpr int NROT = 16;         // rotation warps
  const int G = a.ring_heads, R = a.ring, NB = a.ring_nbuf;
  const int P = a.ring_prod_rows * static_cast<int>(gridDim.x);
  const int p = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x);
  const int rows_p = (CH - p + P - 1) / P;   // rows r = p, p + P, … of every chunk
  const int L = a.seq_len, Lp = a.seq_lp;
  const int total = a.seq_chunks * rows_p;
  const uint32_t box = static_cast<uint32_t>(G) * DK * 2;
  const uint32_t stride = (2 * box + DK * 4 + 1023u) & ~1023u;
  auto buf = [&](int b) { return sb + static_cast<uint32_t>(b) * stride; };
  const uint32_t bars = sb + static_cast<uint32_t>(NB) * stride;
  auto full = [&](int b) { return bars + 8u * static_cast<uint32_t>(b); };
  auto empty = [&](int b) { return bars + 8u * static_cast<uint32_t>(NB + b); };
  uint32_t* ready = a.ring_flags;
  uint32_t* consumed = a.ring_flags + R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < NB; ++b) {
      mbar_init(full(b), 1);
      mbar_init(empty(b), NROT);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == NROT) {
    // ---- loader ----
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = -1;
      for (int n = 0; n < total; ++n) {
        const int b = n % NB;
        if (n >= NB && !mbar_wait(empty(b), static_cast<uint32_t>(n / NB - 1) & 1u, 0x501)) break;
        const int t = (n / rows_p) * CH + p + (n % rows_p) * P;
        if (t < L) {
          mbar_arrive_expect_tx(full(b), 2 * box + DK * 4);
          tma_load_3d_hint(buf(b), tm_rq, 0, t, a.ring_bh0, full(b), pol);
          tma_load_3d_hint(buf(b) + box, tm_rk, 0, t, a.ring_bh0, full(b), pol);
          bulk_load_1d(buf(b) + 2 * box, a.ring_cs + static_cast<size_t>(t) * (DK / 2), DK * 4, full(b));
        } else {
          mbar_arrive(full(b));   // a padding row: nothing to load
        }
        issued = n;
      }
      // Never leave with copies still landing in this CTA's shared memory.
      if (status_aborted())
        for (int n = issued - NB + 1 > 0 ? issued - NB + 1 : 0; n <= issued; ++n)
          mbar_wait(full(n % NB), static_cast<uint32_t>(n / NB) & 1u, 0x5f0, kWaitBudgetCycles / 16);
    }
  } else if (warp < NROT) {
    // ---- rotation ----
    const int cidx = lane % VECS, hsub = lane / VECS;
    bool alive = true;
    for (int n = 0; n < total; ++n) {
      const int b = n % NB;
      const int c = n / rows_p, ri = n % rows_p;
      const int r = p + ri * P, t = c * CH + r, slot = c % R;
      if (alive && ri == 0) {   // this CTA's first row of chunk c: is the slot free?
        int ok = 1;
        if (lane == 0)
          ok = wait_flag_ge(consumed + slot, static_cast<uint32_t>(a.ring_npairs) * static_cast<uint32_t>(c / R),
                            0x502) ? 1 : 0;
        alive = __shfl_sync(0xffffffffu, ok, 0) != 0;
      }
      if (alive) alive = mbar_wait(full(b), static_cast<uint32_t>(n / NB) & 1u, 0x503);
      if (alive) {
        const uint32_t base = buf(b);
        float cv[4] = {0.f, 0.f, 0.f, 0.f}, sv[4] = {0.f, 0.f, 0.f, 0.f};
        if (t < L && !rp.on) {   // the call's table (rows with their own start: below)
          const uint4 c01 = ld_shared_v4(base + 2 * box + cidx * 32);
          const uint4 c23 = ld_shared_v4(base + 2 * box + cidx * 32 + 16);
          cv[0] = __uint_as_float(c01.x); sv[0] = __uint_as_float(c01.y);
          cv[1] = __uint_as_float(c01.z); sv[1] = __uint_as_float(c01.w);
          cv[2] = __uint_as_float(c23.x); sv[2] = __uint_as_float(c23.y);
          cv[3] = __uint_as_float(c23.z); sv[3] = __uint_as_float(c23.w);
        }
        for (int hl = warp * HPW + hsub; hl < G; hl += NROT * HPW) {
          const size_t dst = ((static_cast<size_t>(hl) * R + slot) * CH + r) * DK + 8 * cidx;
          uint4 qo = make_uint4(0u, 0u, 0u, 0u), ko = make_uint4(0u, 0u, 0u, 0u);
          if (t < L) {
            if (rp.on) {   // one start position per batch row: angles of this head's row
              const float pos = rp.p[(a.ring_bh0 + hl) / a.H] + static_cast<float>(t);
#pragma unroll
              for (int u = 0; u < 4; ++u) angle_cs(pos, cc.theta[4 * cidx + u], cv[u], sv[u]);
            }
            float zk, wq;
            row_factors(cc, (a.ring_bh0 + hl) % a.H, t, L, Lp, CH, 1, zk, wq);
            const uint4 qv = ld_shared_v4(base + static_cast<uint32_t>(hl) * DK * 2 + cidx * 16);
            const uint4 kv = ld_shared_v4(base + box + static_cast<uint32_t>(hl) * DK * 2 + cidx * 16);
            qo = make_uint4(rot_q_word(qv.x, cv[0], sv[0], wq), rot_q_word(qv.y, cv[1], sv[1], wq),
                            rot_q_word(qv.z, cv[2], sv[2], wq), rot_q_word(qv.w, cv[3], sv[3], wq));
            ko = make_uint4(rot_k_word(kv.x, __fmul_rn(zk, cv[0]), __fmul_rn(zk, sv[0])),
                            rot_k_word(kv.y, __fmul_rn(zk, cv[1]), __fmul_rn(zk, sv[1])),
                            rot_k_word(kv.z, __fmul_rn(zk, cv[2]), __fmul_rn(zk, sv[2])),
                            rot_k_word(kv.w, __fmul_rn(zk, cv[3]), __fmul_rn(zk, sv[3])));
          }
          *reinterpret_cast<uint4*>(a.ring_q + dst) = qo;
          *reinterpret_cast<uint4*>(a.ring_k + dst) = ko;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(b));
      }
      if (ri == rows_p - 1) {   // this CTA's last row of chunk c: publish the slot
        fence_proxy_async_global();
        named_bar_sync(1, NROT * 32);
        if (threadIdx.x == 0 && !status_aborted()) red_release_gpu_add(ready + slot, 1);
      }
    }
  }
}

// grid = (d_v / 128, rows), cluster = (2, 1, 1); block = 576 threads.
// Warp 0: TMA producer (both CTAs).  Warp 1: pair MMA issuer (even CTA).
// Warps 2..17: drain warps, as in the single-CTA kernel.
// RING: the compact-workspace instantiation (producer CTAs in the first
// grid rows, Q′ / K̂′ read from the ring); without it none of that code is
// compiled in, so the front-pass path keeps its own register allocation.
// MODE: the one-CTA kernel's mode bits (kModeBwd, kModeRev, kModeFold); the
// plain forward instantiation (MODE = 0) compiles none of them.
template <int DK, bool RING, int MODE = 0>
__global__ void __launch_bounds__(NTHREADS, 1)
    pair_tc_kernel(const __grid_constant__ CUtensorMap tm_qh,   // Q′, 64-row boxes
                   const __grid_constant__ CUtensorMap tm_kh,   // K̂′, 64-row boxes
                   const __grid_constant__ CUtensorMap tm_k,    // K̂′, 128-row boxes
                   const __grid_constant__ CUtensorMap tm_v,    // V, 128-row boxes
                   const __grid_constant__ CUtensorMap tm_rq,   // ring mode: raw q, boxes d_k × 1 × heads
                   const __grid_constant__ CUtensorMap tm_rk,   // ring mode: raw k
                   ChunkArgs args, CallConsts cc, RowPos rp) {
  using C = Cfg<DK>;
  constexpr bool BWD = (MODE & tcc::kModeBwd) != 0, REV = (MODE & tcc::kModeRev) != 0,
                 FOLD = (MODE & tcc::kModeFold) != 0;
  static_assert(!(RING && MODE), "the ring mode is a plain forward mode");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  if constexpr (RING) {
    if (static_cast<int>(blockIdx.y) < args.ring_prod_rows) {
      ring_producer<DK>(&tm_rq, &tm_rk, args, cc, rp, sb);
      return;
    }
  }
  const uint32_t sQ = sb + C::OFF_Q, sKQ = sb + C::OFF_KQ, sKV = sb + C::OFF_KV;
  const uint32_t sV = sb + C::OFF_V, sP = sb + C::OFF_P;
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  // The even CTA's barriers in the cluster window (offsets are preserved).
  const uint32_t lead_bar0 = mapa_shared(bar(0), 0);
  auto lead_bar = [&](int i) -> uint32_t { return lead_bar0 + 8u * static_cast<uint32_t>(i); };

  const uint32_t rank = cluster_ctarank();   // 0: issues the pair MMAs
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v0 = blockIdx.x * VT;
  const int grow = FOLD ? static_cast<int>(blockIdx.y + gridDim.y * blockIdx.z) : static_cast<int>(blockIdx.y);
  if (FOLD && args.grid_rows && grow >= args.grid_rows) return;   // both CTAs of the pair
  const int bh = RING ? args.ring_bh0 + grow - args.ring_prod_rows : grow;
  const int seq = bh / args.seq_div, c0 = bh % args.seq_div;   // sequence; its first chunk here
  // Row of chunk c of this sequence in the rotated Q′ / K̂′ source: the
  // padded workspace, or slot c mod R of the ring.
  auto qrow = [&](int c) -> int {
    if constexpr (RING) return ((seq - args.ring_bh0) * args.ring + c % args.ring) * CH;
    return seq * args.seq_lp + c * CH;
  };
  const int h = seq % args.H;
  const int d_v = args.d_v, nch = args.nchunks;
  // γ^{b_c} of chunk c of the sequence (its last chunk may be shorter)
  auto gch = [&](int c) -> float { return c == args.seq_chunks - 1 ? cc.gtail[h] : cc.gb[h]; };
  // chunk of the sequence handled at step i
  auto cix = [&](int i) -> int { return REV ? nch - 1 - i : c0 + i; };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_qh);
    tma_prefetch_desc(&tm_kh);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int i = 0; i < NBAR_; ++i) {
      const bool from_drain = (i == X_READ || i == P_SMEM || i == DS_FREE || i == SH_READY ||
                               i == X_FREE);
      mbar_init(bar(i), from_drain ? 2 * NCW : 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(sb + C::OFF_TPTR, C::T_COLS);
    tmem_relinquish_pair();
  }
  // Both CTAs' barriers exist before any copy or arrival can target them.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::OFF_TPTR);

  if (warp == 0) {
    // ------------------------------ TMA producer ---------------------------
    // Per chunk, in the order the products need them: the V tile and all
    // keys with this CTA's d_k half (ΔS, first), then Q′ rows of this
    // CTA's query half and its key half with all d_k (QK).  Each buffer is
    // refilled as soon as the last product reading it has finished.
    if (lane == 0) {
      // last chunk whose loads were issued, per buffer (for the abort path)
      int iv = -1, ikv = -1, iq = -1, ikq = -1;
      const int yh = 64 * static_cast<int>(rank);
      const int vseq = BWD && args.v_seqs ? seq % args.v_seqs : seq;   // V's row in its tensor map
      for (int i = 0; i < nch; ++i) {
        const int y = qrow(cix(i));       // row of Q′ / K̂′
        const int yv = cix(i) * CH;       // row of V within the sequence
        const int s = i & 1;
        const uint32_t pp = static_cast<uint32_t>(i - 1) & 1u;
        const uint32_t ps = static_cast<uint32_t>((i >> 1) - 1) & 1u;
        if constexpr (RING) {   // the producers have published this chunk's slot
          const int c = c0 + i;
          if (!wait_flag_ge(args.ring_flags + c % args.ring,
                            static_cast<uint32_t>(args.ring_prod_rows * static_cast<int>(gridDim.x)) *
                                static_cast<uint32_t>(c / args.ring + 1),
                            0x105))
            break;
          fence_proxy_async_global();
        }
        if (i > 1 && !mbar_wait(bar(V_EMPTY0 + s), ps, 0x103)) break;
        if (rank == 0) mbar_arrive_expect_tx(bar(V_FULL0 + s), 2 * C::V_BYTES);
        for (int b = 0; b < 2; ++b)
          tma_load_3d_pair(sV + s * C::V_BYTES + b * C::BOX, &tm_v, v0 + 64 * b, yv, vseq, lead_bar(V_FULL0 + s));
        iv = i;
        if (i > 0 && !mbar_wait(bar(KV_EMPTY), pp, 0x104)) break;
        if (rank == 0) mbar_arrive_expect_tx(bar(KV_FULL), 2 * C::KV_BYTES);
        for (int b = 0; b < C::QBOX / 2; ++b)
          tma_load_2d_pair(sKV + b * C::BOX, &tm_k, 64 * (static_cast<int>(rank) * (C::QBOX / 2) + b), y,
                           lead_bar(KV_FULL));
        ikv = i;
        if (i > 1 && !mbar_wait(bar(Q_EMPTY0 + s), ps, 0x102)) break;
        if (rank == 0) mbar_arrive_expect_tx(bar(Q_FULL0 + s), 2 * C::QH_BYTES);
        for (int b = 0; b < C::QBOX; ++b)
          tma_load_2d_pair(sQ + s * C::QH_BYTES + b * C::HBOX, &tm_qh, 64 * b, y + yh, lead_bar(Q_FULL0 + s));
        iq = i;
        if (i > 0 && !mbar_wait(bar(KQ_EMPTY), pp, 0x101)) break;
        if (rank == 0) mbar_arrive_expect_tx(bar(KQ_FULL), 2 * C::KQ_BYTES);
        for (int b = 0; b < C::QBOX; ++b)
          tma_load_2d_pair(sKQ + b * C::HBOX, &tm_kh, 64 * b, y + yh, lead_bar(KQ_FULL));
        ikq = i;
      }
      // Never leave with copies still landing: the even CTA's FULL barriers
      // count both CTAs' bytes, so it waits (bounded) for the last phase of
      // every buffer that was loaded (and of the other slot of the doubled ones).
      if (rank == 0 && status_aborted()) {
        constexpr long long kB = kWaitBudgetCycles / 16;
        for (int c = iv > 0 ? iv - 1 : 0; c <= iv; ++c)
          mbar_wait(bar(V_FULL0 + (c & 1)), static_cast<uint32_t>(c >> 1) & 1u, 0x1f3, kB);
        for (int c = iq > 0 ? iq - 1 : 0; c <= iq; ++c)
          mbar_wait(bar(Q_FULL0 + (c & 1)), static_cast<uint32_t>(c >> 1) & 1u, 0x1f2, kB);
        if (ikv >= 0) mbar_wait(bar(KV_FULL), static_cast<uint32_t>(ikv) & 1u, 0x1f4, kB);
        if (ikq >= 0) mbar_wait(bar(KQ_FULL), static_cast<uint32_t>(ikq) & 1u, 0x1f1, kB);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer -----------------------------
    if (lane == 0 && rank == 0) {
      const uint32_t tX = tmem + C::T_X, tD = tmem + C::T_D, tSH = tmem + C::T_SH;
      constexpr uint32_t ID_P = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t ID_KV = idesc_bf16_f32(256, DK, 1, 1);
      constexpr uint32_t ID_QS = idesc_bf16_f32(256, 128, 0, 0);
      constexpr uint32_t ID_PV = idesc_bf16_f32(256, 128, 1, 0);
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024);                  // K-major, 64 rows
      const uint64_t dQ1 = sdesc_sw128(sQ + C::QH_BYTES, 16, 1024);
      const uint64_t dKQ = sdesc_sw128(sKQ, 16, 1024);                 // K-major, 64 keys
      const uint64_t dKV = sdesc_sw128(sKV, C::BOX, 1024);             // MN-major, d_k half
      const uint64_t dV0 = sdesc_sw128(sV, C::BOX, 1024);              // MN-major
      const uint64_t dV1 = sdesc_sw128(sV + C::V_BYTES, C::BOX, 1024);
      const uint64_t dP = sdesc_sw128(sP, 16, 1024);                   // K-major, 64 rows
      // k-step s of a K-major tile of 64-row boxes, in 16-byte units
#define RET_PAIR_KMAJ(s) static_cast<uint32_t>((((s) >> 2) * C::HBOX + ((s) & 3) * 32) >> 4)
      // Fully unrolled issue: S is the compile-time step index.  MN-major
      // operands advance 2048 bytes (16 keys) per step.
      uint64_t dQ = dQ0, dV = dV0;
      auto issue_qk = [&](auto S) {
        constexpr int k = decltype(S)::value;
        mma_ss_pair_off<RET_PAIR_KMAJ(k), RET_PAIR_KMAJ(k)>(tX, dQ, dKQ, ID_P, k > 0 ? 1u : 0u);
      };
      auto issue_kv = [&](auto S) {
        constexpr int k = decltype(S)::value;
        mma_ss_pair_off<k * 128, k * 128>(tD, dV, dKV, ID_KV, k > 0 ? 1u : 0u);
      };
      auto issue_qs = [&](auto S) {
        constexpr int k = decltype(S)::value;
        mma_ts_pair_off<RET_PAIR_KMAJ(k)>(tX, tSH + k * 8, dQ, ID_QS, k > 0 ? 1u : 0u);
      };
      auto issue_pv = [&](auto S) {
        constexpr int k = decltype(S)::value;
        mma_ss_pair_off<k * 128, RET_PAIR_KMAJ(k)>(tX, dV, dP, ID_PV, 1u);
      };
#undef RET_PAIR_KMAJ
      for (int i = 0; i < nch; ++i) {
        const int s = i & 1;
        const uint32_t pi = static_cast<uint32_t>(i) & 1u;
        const uint32_t pp = static_cast<uint32_t>(i - 1) & 1u;
        const uint32_t pq = static_cast<uint32_t>(i >> 1) & 1u;
        dQ = s ? dQ1 : dQ0;
        dV = s ? dV1 : dV0;
        // 1. ΔSᵀ = Vᵀ K̂′ into D (needs the previous ΔS read out); issued
        // right after PV of the previous chunk, it runs during that Õ drain
        if (!mbar_wait_cl(bar(KV_FULL), pi, 0x201)) break;
        if (!mbar_wait_cl(bar(V_FULL0 + s), pq, 0x202)) break;
        if (i > 0 && !mbar_wait_cl(bar(DS_FREE), pp, 0x203)) break;
        tc_fence_after();
        static_for<CH / 16>(issue_kv);
        mma_commit_pair(bar(DS_FULL));
        mma_commit_pair(bar(KV_EMPTY));
        // 2. P̂ = Q′ K̂′ᵀ into X (needs Õ of the previous chunk read out)
        if (!mbar_wait_cl(bar(KQ_FULL), pi, 0x204)) break;
        if (!mbar_wait_cl(bar(Q_FULL0 + s), pq, 0x205)) break;
        if (i > 0 && !mbar_wait_cl(bar(X_FREE), pp, 0x206)) break;
        tc_fence_after();
        if constexpr (RING)   // this pair has loaded chunk c0 + i out of its ring slot
          red_release_gpu_add(args.ring_flags + args.ring + (c0 + i) % args.ring, 1);
        static_for<DK / 16>(issue_qk);
        mma_commit_pair(bar(P_FULL));
        mma_commit_pair(bar(KQ_EMPTY));
        // 3. Õᵀ = Ŝᵀ Q′ᵀ into X (needs P̂ read out and Ŝ of this chunk)
        if (!mbar_wait_cl(bar(X_READ), pi, 0x207)) break;
        if (!mbar_wait_cl(bar(SH_READY), pi, 0x208)) break;
        tc_fence_after();
        static_for<DK / 16>(issue_qs);
        mma_commit_pair(bar(Q_EMPTY0 + s));
        mma_commit_pair(bar(SH_FREE));
        // 4. Õᵀ += Vᵀ P̂ᵀ (needs both P̂ halves in shared memory)
        if (!mbar_wait_cl(bar(P_SMEM), pi, 0x209)) break;
        tc_fence_after();
        static_for<CH / 16>(issue_pv);
        mma_commit_pair(bar(O_FULL));
        mma_commit_pair(bar(V_EMPTY0 + s));
      }
      // All issued MMAs must finish before either CTA releases its TMEM.
      mma_commit_pair(bar(MMA_DONE));
      mbar_wait(bar(MMA_DONE), 0, 0x2ff);
    }
  } else {
    // ------------------------------ drain warps ----------------------------
    const int w = warp - 2;                 // 0..15
    const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
    const int cs = w >> 2;                  // column slice
    const int kr = w >> 2;                  // state k range [kr*SPT, kr*SPT+SPT)
    const int vl = 32 * quarter + lane;     // TMEM lane: local v for Õ / ΔS / Ŝ
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    const size_t sbase = static_cast<size_t>(bh) * DK * d_v + v0 + vl;

    float S[C::SPT];
#pragma unroll
    for (int u = 0; u < C::SPT; ++u)
      S[u] = args.state_in ? args.state_in[sbase + static_cast<size_t>(kr * C::SPT + u) * d_v] : 0.f;
    if constexpr (BWD) {
      if (args.s_in_exp) {
        const float f = gpow(cc.lg2g[h], static_cast<float>(args.s_in_exp));
#pragma unroll
        for (int u = 0; u < C::SPT; ++u) S[u] *= f;
      }
    }

    auto arrive_lead = [&](int b) {
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(bar(b), 0));
    };
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
      arrive_lead(SH_READY);
    };
    write_shat(gch(cix(0)));

    bool ok = true;
    for (int i = 0; i < nch && ok; ++i) {
      const uint32_t pi = static_cast<uint32_t>(i) & 1u;
      const float gi = gch(cix(i));
      // ---- (a) P̂ drain: causal mask, bf16, into this CTA's query half ----
      if (!mbar_wait(bar(P_FULL), pi, 0x301)) { ok = false; break; }
      tc_fence_after();
      {
        // Lane vl holds query row jl of this CTA's half for the keys of half
        // mh (pair M = 128 layout), columns 16·cs … +15 of that half.
        const int jl = vl & 63, mh = vl >> 6;
        const int j = 64 * static_cast<int>(cluster_ctarank()) + jl;   // query row in the chunk
#pragma unroll
        for (int g = 0; g < 2; ++g) {   // two 8-column rounds keep the register peak low
          uint32_t r[8];
          tmem_ld8(tmem + C::T_X + lane_off + 16 * cs + 8 * g, r);
          tmem_ld_wait();
          if (g == 1) {
            tc_fence_before();
            arrive_lead(X_READ);
          }
          uint32_t pk[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int m = 64 * mh + 16 * cs + 8 * g + 2 * u;
            const bool ka = REV ? m >= j : m <= j, kb = REV ? m + 1 >= j : m + 1 <= j;
            const float a = ka ? __uint_as_float(r[2 * u]) : 0.f;
            const float b = kb ? __uint_as_float(r[2 * u + 1]) : 0.f;
            pk[u] = pack_bf16x2(a, b);
          }
          st_shared_v4(sP + mh * C::HBOX + sw128_offset(jl, 16 * cs + 8 * g), pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async_smem();
      arrive_lead(P_SMEM);

      // ---- (b) ΔS drain: S = fmaf(γ^b, S, ΔS) ----
      if (!mbar_wait(bar(DS_FULL), pi, 0x302)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < C::SPT / 16; ++c) {   // 16 columns per wait
        uint32_t d[16];
        tmem_ld16(tmem + C::T_D + lane_off + kr * C::SPT + c * 16, d);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; ++u)
          S[16 * c + u] = args.raw_ds ? __uint_as_float(d[u]) : fmaf(gi, S[16 * c + u], __uint_as_float(d[u]));
      }
      tc_fence_before();
      arrive_lead(DS_FREE);

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
        if (args.out && !args.out_f32) {
          // bf16 output: the first 16 rows packed to bf16 pairs, the last 16
          // loaded, X released, and only then the 32 stores, so that no store
          // sits on the chain Õ drain → QK of the next chunk.
          uint32_t pk[8], r[16];
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs, *reinterpret_cast<uint32_t(*)[8]>(&r[0]));
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 8, *reinterpret_cast<uint32_t(*)[8]>(&r[8]));
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 8; ++u) pk[u] = pack_bf16x2(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 16, *reinterpret_cast<uint32_t(*)[8]>(&r[0]));
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 24, *reinterpret_cast<uint32_t(*)[8]>(&r[8]));
          tmem_ld_wait();
          tc_fence_before();
          arrive_lead(X_FREE);
          unsigned short* o = reinterpret_cast<unsigned short*>(static_cast<__nv_bfloat16*>(obuf) + base);
#pragma unroll
          for (int u = 0; u < 8; ++u) {   // streaming stores: the output is not read again here
            __stcs(o + static_cast<size_t>(2 * u) * d_v, static_cast<unsigned short>(pk[u] & 0xffffu));
            __stcs(o + static_cast<size_t>(2 * u + 1) * d_v, static_cast<unsigned short>(pk[u] >> 16));
          }
#pragma unroll
          for (int c = 0; c < 16; ++c)
            __stcs(o + static_cast<size_t>(16 + c) * d_v,
                   __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[c]))));
        } else
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t r[16];
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 16 * hf, *reinterpret_cast<uint32_t(*)[8]>(&r[0]));
          tmem_ld8(tmem + C::T_X + lane_off + 32 * cs + 16 * hf + 8, *reinterpret_cast<uint32_t(*)[8]>(&r[8]));
          tmem_ld_wait();
          if (hf == 1) {
            tc_fence_before();
            arrive_lead(X_FREE);
          }
          const size_t gb0 = base + static_cast<size_t>(16 * hf) * d_v;
          if (!args.out) {
          } else if (args.out_f32) {
            float* o = reinterpret_cast<float*>(obuf) + gb0;
#pragma unroll
            for (int c = 0; c < 16; ++c) o[static_cast<size_t>(c) * d_v] = __uint_as_float(r[c]);
          } else {
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(obuf) + gb0;
#pragma unroll
            for (int c = 0; c < 16; ++c)   // streaming stores: the output is not read again here
              __stcs(reinterpret_cast<unsigned short*>(o + static_cast<size_t>(c) * d_v),
                     __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[c]))));
          }
        }
      }
    }
    if (ok && args.state_out) {
#pragma unroll
      for (int u = 0; u < C::SPT; ++u)
        args.state_out[sbase + static_cast<size_t>(kr * C::SPT + u) * d_v] =
            BWD && args.s_out_exp ? S[u] * gpow(cc.lg2g[h], static_cast<float>(args.s_out_exp)) : S[u];
    }
  }

  // Neither CTA leaves (or frees its TMEM) while the other may still arrive
  // on its barriers or the pair MMAs may still touch its memory.
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::T_COLS);
  }
}

}  // namespace tcq
}  // namespace ret
