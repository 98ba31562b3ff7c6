// fa_fwd.cu -- exact attention forward for sm_103a.
//
// One CTA owns two query tiles of 128 rows (256 consecutive rows of one head;
// one tile of 128 rows at d = 256) and walks the key/value tiles of 128 rows of
// that head:
//
//   tiling      -- "FlashAttention" wiki note, 定義 item (1); the explainer's
//                  tiling paragraph (blocks loaded from HBM into on-chip memory,
//                  local scores computed there, no N x N matrix in HBM);
//   online softmax with rescale when the running max grows -- the explainer's
//                  online-softmax paragraph;
//   asynchronous MMA, warp specialisation, TMA -- wiki sections FA3 (1), FA4 (1);
//   conditional rescale -- FA4 summary (ai-papers.net), 提案手法 item 2, and the
//                  wiki's FA4 (2): the O/l correction is skipped unless the row
//                  max has grown by more than tau (log2 units) since the value
//                  the exponentials are taken against; the result is exact
//                  because O and l always share that reference max.
//
// Warp roles (320 threads):
//   warps 0-3  softmax for query tile 0 (thread = row = TMEM lane)
//   warps 4-7  softmax for query tile 1
//   warp 8     MMA issuer (one thread) and TMEM allocator
//   warp 9     TMA producer (one thread)
// Tensor memory (512 columns): S0 | S1 | O0 | O1; P (bf16) overwrites the first
// half of its S block and feeds the PV MMA straight from TMEM.
// Shared memory: Q0, Q1 and a ring of K/V tiles (K_j and V_j take turns).
//
// Variants of the same kernel:
//   Nq != Nk     the causal mask places query row i at position i + (Nk - Nq);
//   one tile     a block with at most 128 rows runs query tile 0 only;
//   split-KV     (decoding) several CTAs share a block's key tiles, each writing an
//                fp32 partial O and its LSE, merged by fwd_combine_kernel; the query
//                heads of a K/V group are packed as the rows of one block, each row
//                keeping its own causal position (pos_mod).
#include <algorithm>
#include <type_traits>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

// DEC: the decoding configuration (split-KV units of at most 128 query rows): one query tile,
// 192 threads (one softmax warpgroup, the MMA warp and the TMA warp) and 256 tensor-memory
// columns, so that two CTAs share an SM and their per-tile chains (S MMA -> softmax -> PV MMA)
// overlap; one such chain per SM streams K/V well short of the HBM copy rate.
template <int D, bool DEC = false>
struct FwdCfg {
  static constexpr int BM = 128;                    // rows per query tile
  static constexpr int BN = 128;                    // keys per K/V tile
  static constexpr int TILE = 128 * D * 2;          // bytes of one 128 x D bf16 tile
  static constexpr int CHUNKS = D / 64;             // 128-byte swizzle atoms across D
  // query tiles per work unit: two (S0 | S1 | O0 | O1 in TMEM), or one at d = 256 (S0 | O0
  // already take 384 of the 512 columns)
  static constexpr int NT = (DEC || D == 256) ? 1 : 2;
  static constexpr int BLOCK = 128 * NT;            // query rows per work unit
  static constexpr int STAGES = DEC ? (D == 64 ? 4 : 2) : (D == 256) ? 2 : (D == 128) ? 4 : 8;  // K/V ring slots
  static constexpr int SMEM_Q = NT * TILE;
  static constexpr int SMEM_RING = STAGES * TILE;
  static constexpr int NBAR = 2 * STAGES + 11;
  static constexpr int SMEM_BYTES = 1024 + SMEM_Q + SMEM_RING + NBAR * 8 + 16;
  static constexpr int THREADS = DEC ? 192 : 384;
  static constexpr int SOFT_WARPS = DEC ? 4 : 8;     // softmax warps; the copy/MMA warps follow
  static constexpr int MIN_BLOCKS = DEC ? 2 : 1;     // CTAs per SM
  static constexpr int TMEM_COLS = DEC ? 256 : 512;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = (NT == 2) ? 256 : 128, COL_O1 = 256 + D;
  // d = 256: S | O take 384 columns, so a second S buffer fits (columns 384-511).  Key tiles
  // alternate between the two, so the next tile's S MMAs run while the softmax works on this
  // one; K and V then come from two copy threads, so that a K load never queues behind a V
  // slot the PV MMA still holds.
  static constexpr bool DS = (D == 256 && !DEC);
  static constexpr uint32_t COL_SB = 384;
  // Register split (setmaxnreg): the kernel is launched at 168 registers per thread (384
  // threads, 64512 registers); the two softmax warpgroups take 184 each, the copy/MMA
  // warpgroup keeps 136.  The shares must add up to the launch's total, or the increase waits
  // forever (build.py checks the compiled register count).
  // The decoding configuration (one softmax warpgroup plus the MMA and TMA warps, 192 threads,
  // two CTAs per SM) has no whole second warpgroup and so no split: every thread keeps the 168
  // registers that two CTAs of 192 threads leave.
  static constexpr int REG_LAUNCH = 168, REG_SOFTMAX = DEC ? 168 : 184, REG_OTHER = DEC ? 168 : 136;
  static_assert(DEC || (SOFT_WARPS / 4) * 128 * REG_SOFTMAX + (THREADS / 128 - SOFT_WARPS / 4) * 128 * REG_OTHER ==
                           THREADS * REG_LAUNCH,
                "register split");
  static_assert(!DEC || MIN_BLOCKS * THREADS * REG_LAUNCH <= 65536, "two CTAs per SM");
};

// One work unit: a block of BLOCK query rows of one (b, h) and, with split-KV, a key range.
struct FwdUnit {
  int bh, q0, j0, n_kv, kv_z;
  int sp;    // key-range split (0 when splits = 1)
  bool two;  // the block has rows in query tile 1
};

// Units are numbered heaviest first under a causal mask (the blocks nearest the end of the
// sequence see the most keys), then by (b, h), then by split.
template <int D, bool DEC = false>
FA_DEV FwdUnit fwd_unit(const FwdParams& p, int u) {
  using C = FwdCfg<D, DEC>;
  const int N = p.Nq;  // query rows; keys: p.Nk
  const int ncb = (N + C::BLOCK - 1) / C::BLOCK;
  const int BH = p.B * p.H;
  FwdUnit w;
  w.sp = u % p.splits;
  const int t = u / p.splits;
  const int cb = p.causal ? (ncb - 1 - t / BH) : (t / BH);
  w.bh = t % BH;
  const int b = w.bh / p.H, h = w.bh % p.H;
  const int g = h / (p.H / p.Hkv);
  w.q0 = cb * C::BLOCK;
  const int n_kv_all = (p.Nk + 127) / 128;
  // causal: the block's last row (position row + qoff) bounds the key tiles it needs; a block
  // whose rows see no key at all still runs one fully masked tile (O = 0, LSE = -inf)
  const int last_row = min(w.q0 + C::BLOCK - 1, N - 1);
  const int k_last = (p.pos_mod ? min(last_row, p.pos_mod - 1) : last_row) + p.qoff;
  const int n_vis = p.causal ? (k_last < 0 ? 1 : min(n_kv_all, k_last / 128 + 1)) : n_kv_all;
  // this unit's key tiles [j0, j0 + n_kv); a split whose range holds no visible key still runs
  // one fully masked tile, which gives O = 0 and LSE = -inf for it
  w.j0 = w.sp * p.split_tiles;
  w.n_kv = max(1, min(n_vis, w.j0 + p.split_tiles) - w.j0);
  // a block with at most 128 rows (a ragged last block; decoding) runs query tile 0 only
  w.two = C::NT == 2 && N - w.q0 > 128;
  w.kv_z = b * p.Hkv + g;
  return w;
}

// The r-th unit of this CTA: one CTA per SM walks the units in boustrophedon order (row r of
// gridDim.x units left to right when r is even, right to left when odd), which balances the
// heaviest-first causal costs across CTAs to within about 1% on large problems.
FA_DEV int fwd_unit_index(int r) {
  const int G = gridDim.x;
  return r * G + ((r & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
}

// POLY: how many of every 16 column pairs take the FMA-pipe polynomial exp2 instead of
// the MUFU ex2 unit (0 = MUFU only).
template <int D, int POLY, bool DEC = false>
__global__ void __launch_bounds__(FwdCfg<D, DEC>::THREADS, FwdCfg<D, DEC>::MIN_BLOCKS)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p, int n_units) {
  using C = FwdCfg<D, DEC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::SMEM_Q;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sRing + C::SMEM_RING);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  const uint32_t q_full = bar0 + 8u * (2 * C::STAGES);
  const uint32_t q_empty = bar0 + 8u * (2 * C::STAGES + 1);
  auto s_full = [&](int w) { return bar0 + 8u * (2 * C::STAGES + 2 + w); };
  auto p_full = [&](int w) { return bar0 + 8u * (2 * C::STAGES + 4 + w); };
  auto o_bar = [&](int w) { return bar0 + 8u * (2 * C::STAGES + 6 + w); };
  auto o_free = [&](int w) { return bar0 + 8u * (2 * C::STAGES + 8 + w); };
  const uint32_t mma_done = bar0 + 8u * (2 * C::STAGES + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const Abort ab{abort, p.status, p.kabort, p.gen};

  const int warp = warp_id();
  const int lane = lane_id();
  const int N = p.Nq;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int w = 0; w < 2; ++w) {
      mbar_init(s_full(w), 1);
      mbar_init(p_full(w), 128);
      mbar_init(o_bar(w), 1);
      mbar_init(o_free(w), 128);
    }
    mbar_init(mma_done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == C::SOFT_WARPS) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == C::SOFT_WARPS + 1 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= C::SOFT_WARPS) {
    if constexpr (!DEC) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_OTHER));
    if ((warp == C::SOFT_WARPS + 1 || (C::DS && warp == C::SOFT_WARPS + 2)) && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      // (with two S buffers: warp SOFT_WARPS + 1 loads Q and K, warp SOFT_WARPS + 2 loads V)
      const bool do_k = !C::DS || warp == C::SOFT_WARPS + 1;
      const bool do_v = !C::DS || warp == C::SOFT_WARPS + 2;
      uint32_t it = 0;      // ring position of the next K/V load (continues across units)
      uint32_t issued = 0;  // ring loads issued
      int q_loads = 0;   // Q loads issued (one per unit)
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int u = fwd_unit_index(r);
        if (u >= n_units) break;
        const FwdUnit w = fwd_unit<D, DEC>(p, u);
        if (do_k) {
          // the Q buffer is free once the previous unit's last S MMAs have completed
          if (q_loads > 0 && !mbar_wait(q_empty, (q_loads - 1) & 1, ab)) break;
          mbar_arrive_expect_tx(q_full, C::NT * C::TILE);
          for (int qt = 0; qt < C::NT; ++qt)
            for (int ch = 0; ch < C::CHUNKS; ++ch)
              tma_load_3d(smem_u32(sQ + qt * C::TILE + ch * 16384), &tm_q, q_full, ch * 64, w.q0 + qt * 128, w.bh);
          ++q_loads;
        }
        for (int jj = 0; jj < 2 * w.n_kv; ++jj, ++it) {
          const int slot = it % C::STAGES;
          if (!((jj & 1) ? do_v : do_k)) continue;  // the other copy thread's load
          if (r == 0 && jj == p.drop_it) continue;  // failure-injection test hook (never set in normal use)
          if (!mbar_wait(empty_bar(slot), ((it / C::STAGES) & 1) ^ 1, ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(slot), C::TILE);
          for (int ch = 0; ch < C::CHUNKS; ++ch)
            tma_load_3d(smem_u32(sRing + slot * C::TILE + ch * 16384), (jj & 1) ? &tm_v : &tm_k, full_bar(slot),
                        ch * 64, (w.j0 + (jj >> 1)) * 128, w.kv_z);
          issued = it + 1;
        }
      }
      if (*abort) {
        // The CTA gave up: let the copies still in flight land before the CTA exits (each
        // completes its slot's phase), bounded at 1 ms per copy.
        for (uint32_t k = issued > C::STAGES ? issued - C::STAGES : 0; k < issued; ++k) {
          if (!((k & 1) ? do_v : do_k)) continue;  // (two S buffers: the other thread's load)
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(full_bar(k % C::STAGES), (k / C::STAGES) & 1) && globaltimer() - t0 < 1000000ull) {
          }
        }
        if (q_loads > 0) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(q_full, (q_loads - 1) & 1) && globaltimer() - t0 < 1000000ull) {
          }
        }
      }
    } else if (warp == C::SOFT_WARPS && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t ring = smem_u32(sRing);
      auto issue_s = [&](int w, int slot) {
        const uint32_t a0 = q_addr + w * C::TILE, b0 = ring + slot * C::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + (w ? C::COL_S1 : C::COL_S0), sdesc_sw128(a0 + off, 16, 1024), sdesc_sw128(b0 + off, 16, 1024),
                 idS, kk > 0);
        }
      };
      auto issue_pv = [&](int w, int slot, bool acc) {
        const uint32_t v0 = ring + slot * C::TILE;
        const uint32_t sc = w ? C::COL_S1 : C::COL_S0;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + (w ? C::COL_O1 : C::COL_O0), tmem + sc + kk * 8, sdesc_sw128(v0 + kk * 2048, 16384, 1024),
                 idO, (acc || kk > 0) ? 1u : 0u);
      };
      // two S buffers (d = 256): Q against K in `slot` into the S columns `col`; O += P V
      // with P read from the S columns `col`
      auto issue_s_col = [&](uint32_t col, int slot) {
        const uint32_t b0 = ring + slot * C::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + col, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(b0 + off, 16, 1024), idS, kk > 0);
        }
      };
      auto issue_pv_col = [&](uint32_t col, int slot, bool acc) {
        const uint32_t v0 = ring + slot * C::TILE;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::COL_O0, tmem + col + kk * 8, sdesc_sw128(v0 + kk * 2048, 16384, 1024), idO,
                 (acc || kk > 0) ? 1u : 0u);
      };
      auto slot_of = [](uint32_t k) { return k % C::STAGES; };
      auto par_of = [](uint32_t k) { return (k / C::STAGES) & 1u; };
      uint32_t it = 0;          // ring position (continues across units)
      uint32_t units = 0;       // units issued (q_full phase, o_free(0) phase)
      uint32_t units2 = 0;      // two-tile units issued (o_free(1) phase)
      uint32_t jg0 = 0, jg1 = 0;  // key tiles issued per query tile (p_full phases)
      // One unit's MMAs, compiled once for two query tiles and once for one: a run-time branch
      // on the tile count inside this one-lane issue loop costs about 1% of the kernel.  The
      // loop reads only values fixed for the unit (ring base, phase bases), so nothing it
      // needs is written inside it.
      auto unit_mma = [&](const FwdUnit& w, auto two_tiles, const uint32_t it0, const uint32_t u_idx,
                          const uint32_t u2_idx, const uint32_t g0, const uint32_t g1) -> bool {
        constexpr bool TWO = decltype(two_tiles)::value;
        const int n_kv = w.n_kv;
        if constexpr (C::DS) {
          // Key tile G (counted over the CTA's units) uses S buffer G & 1 and the barriers
          // s_full / p_full / o_bar of that buffer.  S(G + 1) is issued before the wait for P(G),
          // so it runs while the softmax works on tile G; P(G) in buffer G & 1 is read by PV(G)
          // before S(G + 2) overwrites it (MMAs complete in issue order).
          auto scol = [](uint32_t G) { return (G & 1) ? C::COL_SB : C::COL_S0; };
          if (!mbar_wait(q_full, u_idx & 1, ab)) return false;
          if (!mbar_wait(full_bar(slot_of(it0)), par_of(it0), ab)) return false;
          tc_fence_after();
          issue_s_col(scol(g0), slot_of(it0));
          mma_commit(s_full(g0 & 1));
          if (n_kv == 1) mma_commit(q_empty);
          mma_commit(empty_bar(slot_of(it0)));
          if (u_idx > 0 && !mbar_wait(o_free(0), (u_idx - 1) & 1, ab)) return false;
          for (int j = 0; j < n_kv; ++j) {
            const uint32_t G = g0 + j;
            if (j + 1 < n_kv) {
              const uint32_t itk = it0 + 2 * (j + 1);
              if (!mbar_wait(full_bar(slot_of(itk)), par_of(itk), ab)) return false;
              tc_fence_after();
              issue_s_col(scol(G + 1), slot_of(itk));
              mma_commit(s_full((G + 1) & 1));
              if (j + 2 == n_kv) mma_commit(q_empty);
              mma_commit(empty_bar(slot_of(itk)));
            }
            const uint32_t itv = it0 + 2 * j + 1;
            if (!mbar_wait(full_bar(slot_of(itv)), par_of(itv), ab)) return false;
            if (!mbar_wait(p_full(G & 1), (G >> 1) & 1, ab)) return false;
            tc_fence_after();
            issue_pv_col(scol(G), slot_of(itv), j > 0);
            mma_commit(o_bar(G & 1));
            mma_commit(empty_bar(slot_of(itv)));
          }
          return true;
        }
        if (!mbar_wait(q_full, u_idx & 1, ab)) return false;
        if (!mbar_wait(full_bar(slot_of(it0)), par_of(it0), ab)) return false;
        tc_fence_after();
        issue_s(0, slot_of(it0));
        mma_commit(s_full(0));
        if constexpr (TWO) {
          issue_s(1, slot_of(it0));
          mma_commit(s_full(1));
        }
        if (n_kv == 1) mma_commit(q_empty);  // the unit's last S MMAs: the Q buffer frees after them
        mma_commit(empty_bar(slot_of(it0)));
        // The first PV of a query tile overwrites its O accumulator, which the softmax warps
        // of the previous unit may still be reading out; they release it before they start on
        // this unit's first exponentials, so this wait rarely stalls.
        if (u_idx > 0 && !mbar_wait(o_free(0), (u_idx - 1) & 1, ab)) return false;
        if constexpr (TWO) {
          if (u2_idx > 0 && !mbar_wait(o_free(1), (u2_idx - 1) & 1, ab)) return false;
        }
        // one key tile; MORE: another tile follows (the last iteration is peeled so that the
        // test is not a run-time branch of the issue loop)
        auto step = [&](int j, auto more_tiles) -> bool {
          constexpr bool MORE = decltype(more_tiles)::value;
          const uint32_t itv = it0 + 2 * j + 1, itk = itv + 1;
          if (!mbar_wait(full_bar(slot_of(itv)), par_of(itv), ab)) return false;
          if (!mbar_wait(p_full(0), (g0 + j) & 1, ab)) return false;
          tc_fence_after();
          issue_pv(0, slot_of(itv), j > 0);
          mma_commit(o_bar(0));
          if constexpr (MORE) {
            if (!mbar_wait(full_bar(slot_of(itk)), par_of(itk), ab)) return false;
            tc_fence_after();
            issue_s(0, slot_of(itk));
            mma_commit(s_full(0));
          }
          if constexpr (TWO) {
            if (!mbar_wait(p_full(1), (g1 + j) & 1, ab)) return false;
            tc_fence_after();
            issue_pv(1, slot_of(itv), j > 0);
            mma_commit(o_bar(1));
          }
          mma_commit(empty_bar(slot_of(itv)));
          if constexpr (MORE) {
            if constexpr (TWO) {
              issue_s(1, slot_of(itk));
              mma_commit(s_full(1));
            }
            if (j + 2 == n_kv) mma_commit(q_empty);
            mma_commit(empty_bar(slot_of(itk)));
          }
          return true;
        };
        bool ok = true;
        for (int j = 0; ok && j + 1 < n_kv; ++j) ok = step(j, std::true_type{});
        if (ok) ok = step(n_kv - 1, std::false_type{});
        return ok;
      };
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int u = fwd_unit_index(r);
        if (u >= n_units) break;
        const FwdUnit w = fwd_unit<D, DEC>(p, u);
        ok = w.two ? unit_mma(w, std::true_type{}, it, units, units2, jg0, jg1)
                   : unit_mma(w, std::false_type{}, it, units, units2, jg0, jg1);
        it += 2 * w.n_kv;
        jg0 += w.n_kv;
        ++units;
        if (w.two) {
          jg1 += w.n_kv;
          ++units2;
        }
      }
      // drain: every MMA issued above has finished before TMEM is released (bounded, and
      // waited for even after an abort)
      mma_commit(mma_done);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(mma_done, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    if constexpr (!DEC) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_SOFTMAX));
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int w = warp >> 2;            // query tile
    const int r = threadIdx.x & 127;    // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (w ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = tmem + lane_off + (w ? C::COL_O1 : C::COL_O0);
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const int BH = p.B * p.H;
    int jg = 0;  // key tiles processed by this warpgroup (s_full, o_bar phases)
    bool ok = true;
    for (int ru = 0; ok; ++ru) {
      const int u = fwd_unit_index(ru);
      if (u >= n_units) break;
      const FwdUnit wu = fwd_unit<D, DEC>(p, u);
      if (w == 1 && !wu.two) continue;  // no row of this block falls in query tile 1
      const int row = wu.q0 + w * 128 + r;                 // absolute query row
      const int rpos = p.pos_mod ? row % p.pos_mod : row;  // its position for the causal mask
      float m_used = -INFINITY;      // reference max (log2 units) of O and l
      uint64_t l_exact = 0;          // sum of p (fp32 pair): gives the LSE
      // sum of bf16(p), the weights the PV MMA used: normalises O.  Two accumulators, each
      // taking both halves of every other packed pair through mixed-precision adds (fewer
      // instructions and shorter dependency chains than widening the pairs: 0.900 -> 0.864 ms
      // on the B4 H16 N8192 causal workload)
      float lr0 = 0.f, lr1 = 0.f;
      const int tile_row0 = wu.q0 + w * 128;
      for (int j = 0; j < wu.n_kv; ++j, ++jg) {
        // (two S buffers: key tile jg uses buffer jg & 1 and that buffer's barriers)
        const int sb = C::DS ? (jg & 1) : w;
        const uint32_t tSj = C::DS ? (tmem + lane_off + ((jg & 1) ? C::COL_SB : C::COL_S0)) : tS;
        ok = __all_sync(0xffffffffu, mbar_wait(s_full(sb), C::DS ? ((jg >> 1) & 1) : (jg & 1), ab));
        if (!ok) break;
        tc_fence_after();
        const int col0 = (wu.j0 + j) * 128;
        // column c of the tile is masked from lim on: past Nk, or (causal) after the row's position
        const int lim = p.causal ? min(p.Nk - col0, rpos + p.qoff + 1 - col0) : p.Nk - col0;
        // whether the tile needs the mask at all (a test on the tile's first row, or at d = 64, on
        // the warp's rows: the forms that keep each instantiation free of register spills)
        bool mask_tile;
        if constexpr (D == 64) {
          mask_tile = __any_sync(0xffffffffu, lim < 128);
        } else {  // packed rows: the smallest position in the tile is 0 (+ qoff)
          mask_tile = (p.causal && col0 + 127 > (p.pos_mod ? 0 : tile_row0) + p.qoff) || col0 + 128 > p.Nk;
        }
        float s[128];
        {
          uint32_t rr[128];
          tmem_ld128(tSj, rr);  // one load and one wait for the whole row
#pragma unroll
          for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(rr[i]);
        }
        if (mask_tile) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) s[c] = -INFINITY;
        }
        float mx4[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          float m = fmaxf(s[32 * a], s[32 * a + 1]);
#pragma unroll
          for (int c = 2; c < 32; c += 2) m = max3f(m, s[32 * a + c], s[32 * a + c + 1]);
          mx4[a] = m;
        }
        const float mx = fmaxf(max3f(mx4[0], mx4[1], mx4[2]), mx4[3]);
        const float m_tile = mx * sl2;
        const bool need = m_tile > m_used + p.tau;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? m_tile : m_used;
          const float alpha = need ? ex2_mufu(m_used - m_new) : 1.f;
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            if (p.rescale_events) {  // debug counter: rows whose O is rescaled at this key tile
              const unsigned moved = __ballot_sync(0xffffffffu, alpha != 1.f);
              if (lane == 0) atomicAdd(p.rescale_events, (unsigned long long)__popc(moved));
            }
            // O holds sum_{j'<j} P V against m_used; it must be complete before rescaling
            // (two S buffers: the previous tile's PV commits to its buffer's o_bar)
            ok = __all_sync(0xffffffffu, mbar_wait(o_bar(C::DS ? ((jg - 1) & 1) : w),
                                                   C::DS ? (((jg - 1) >> 1) & 1) : ((jg - 1) & 1), ab));
            if (!ok) break;
            tc_fence_after();
            auto rescale16 = [&](int c) {
              uint32_t rr[16];
              tmem_ld16(tO + 16 * c, rr);
#pragma unroll
              for (int i = 0; i < 16; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
              tmem_st16(tO + 16 * c, rr);
            };
            if constexpr (D == 256) {
              // a rolled loop: with the whole score row live, an unrolled one spills at d = 256
#pragma unroll 1
              for (int c = 0; c < D / 16; ++c) rescale16(c);
            } else {
#pragma unroll
              for (int c = 0; c < D / 16; ++c) rescale16(c);
            }
            tmem_st_wait();
          }
          const uint64_t a2 = f2_pack(alpha, alpha);
          l_exact = f2_mul(l_exact, a2);
          lr0 *= alpha;
          lr1 *= alpha;
          m_used = m_new;
        }
        const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
        const uint64_t nm2 = f2_pack(neg_m, neg_m);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t x2 = f2_fma(f2_pack(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), sl2x2, nm2);
            float p0, p1;
            if ((i * POLY) % 16 < POLY) {
              const float2 pp = f2_unpack(ex2_poly2(x2));
              p0 = pp.x;
              p1 = pp.y;
            } else {
              const float2 x = f2_unpack(x2);
              p0 = ex2_mufu(x.x);
              p1 = ex2_mufu(x.y);
            }
            pk[i] = pack_bf16x2(p0, p1);
            l_exact = f2_add(l_exact, f2_pack(p0, p1));
            if (i & 1)
              lr1 = add_bf16_hi(add_bf16_lo(lr1, pk[i]), pk[i]);
            else
              lr0 = add_bf16_hi(add_bf16_lo(lr0, pk[i]), pk[i]);
          }
          tmem_st16(tSj + 16 * c, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full(sb));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, LSE = ln 2 * (m_used + log2 l).  O's tensor memory is
      // handed back (o_free) right after the last load from it, so the next unit's first PV
      // MMA can overwrite it while these stores drain.
      ok = __all_sync(0xffffffffu, mbar_wait(o_bar(C::DS ? ((jg - 1) & 1) : w),
                                             C::DS ? (((jg - 1) >> 1) & 1) : ((jg - 1) & 1), ab));
      if (!ok) break;
      tc_fence_after();
      const float2 le = f2_unpack(l_exact);
      const float l = le.x + le.y, lrs = lr0 + lr1;
      const float inv_l = lrs > 0.f ? 1.f / lrs : 0.f;
      if (p.splits > 1) {  // split-KV partial: fp32 O over this split's keys, LSE in log2 units
        const size_t prow = ((size_t)wu.sp * BH + wu.bh) * N + row;
        float4* op = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(tO + 32 * c, rr);
          if (c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(o_free(w));
          }
          if (row < N) {
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              op[c * 8 + v4] = make_float4(__uint_as_float(rr[4 * v4]) * inv_l, __uint_as_float(rr[4 * v4 + 1]) * inv_l,
                                           __uint_as_float(rr[4 * v4 + 2]) * inv_l, __uint_as_float(rr[4 * v4 + 3]) * inv_l);
          }
        }
        if (row < N) p.lse_part[prow] = l > 0.f ? m_used + log2f(l) : -INFINITY;
      } else {
        uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + ((size_t)wu.bh * N + row) * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(tO + 32 * c, rr);
          if (c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(o_free(w));
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * inv_l, __uint_as_float(rr[2 * i + 1]) * inv_l);
          if (row < N) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              orow[c * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        if (row < N) p.lse[(size_t)wu.bh * N + row] = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::SOFT_WARPS) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

static int fwd_sm_count() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 148;
  }
  return n[dev];
}

template <int D, int POLY, bool DEC = false>
static cudaError_t launch_fwd_dp(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D, DEC>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(fwd_kernel<D, POLY, DEC>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const long long units = (long long)((p.Nq + C::BLOCK - 1) / C::BLOCK) * p.B * p.H * p.splits;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  // persistent: one CTA per SM (two in the decoding configuration), at most one per unit
  const int grid = (int)std::min<long long>(units, (long long)fwd_sm_count() * C::MIN_BLOCKS);
  fwd_kernel<D, POLY, DEC><<<dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(tq, tk, tv, p, (int)units);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdParams& p, int poly_cols, cudaStream_t stream) {
  switch (poly_cols) {  // columns of every 32 on the polynomial
    case 0: return launch_fwd_dp<D, 0>(tq, tk, tv, p, stream);
    case 4: return launch_fwd_dp<D, 2>(tq, tk, tv, p, stream);
    case 8: return launch_fwd_dp<D, 4>(tq, tk, tv, p, stream);
    case 12: return launch_fwd_dp<D, 6>(tq, tk, tv, p, stream);
    case 16: return launch_fwd_dp<D, 8>(tq, tk, tv, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

bool fwd_decoding_config(int d, int rows, int splits, int poly_cols) {
  return (d == 64 || d == 128) && poly_cols == 0 && splits > 1 && rows <= 128;
}

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int poly_cols, cudaStream_t stream) {
  if (fwd_decoding_config(d, p.Nq, p.splits, poly_cols))
    return d == 64 ? launch_fwd_dp<64, 0, true>(tq, tk, tv, p, stream) : launch_fwd_dp<128, 0, true>(tq, tk, tv, p, stream);
  if (d == 64) return launch_fwd_d<64>(tq, tk, tv, p, poly_cols, stream);
  if (d == 256) {  // MUFU exponentials only at d = 256
    if (poly_cols != 0) return cudaErrorInvalidValue;
    return launch_fwd_dp<256, 0>(tq, tk, tv, p, stream);
  }
  return launch_fwd_d<128>(tq, tk, tv, p, poly_cols, stream);
}

// Split-KV merge, one warp per query row: with m = max_s lse_s (log2 units) and
// w_s = 2^(lse_s - m), O = sum_s w_s o_s / sum_s w_s and LSE = ln 2 * (m + log2 sum_s w_s) —
// the online-softmax merge of the splits' (max, sum, output) triples.
template <int D>
__global__ void __launch_bounds__(256) fwd_combine_kernel(const float* __restrict__ o_part,
                                                          const float* __restrict__ lse_part, uint16_t* __restrict__ o,
                                                          float* __restrict__ lse, int S, long long rows) {
  constexpr int PER = D / 32;  // fp32 elements per lane (2, 4 or 8)
  const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
  const int lane = threadIdx.x & 31;
  for (long long row = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); row < rows; row += nwarps) {
    float m = -INFINITY;
    for (int s = lane; s < S; s += 32) m = fmaxf(m, lse_part[(size_t)s * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float acc[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) acc[k] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < S; ++s) {
        const float ls = lse_part[(size_t)s * rows + row];
        const float wgt = ls == -INFINITY ? 0.f : exp2f(ls - m);
        wsum += wgt;
        const float* src = o_part + ((size_t)s * rows + row) * D + lane * PER;
#pragma unroll
        for (int k = 0; k < PER; ++k) acc[k] = fmaf(wgt, src[k], acc[k]);
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint16_t* dst = o + row * D + lane * PER;
#pragma unroll
    for (int k = 0; k < PER; k += 2) {
      const uint32_t pk = pack_bf16x2(acc[k] * inv, acc[k + 1] * inv);
      *reinterpret_cast<uint32_t*>(dst + k) = pk;
    }
    if (lane == 0) lse[row] = wsum > 0.f ? (m + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
  }
}

cudaError_t launch_fwd_combine(int d, const float* o_part, const float* lse_part, void* o, float* lse, int splits,
                               long long rows, cudaStream_t stream) {
  const long long want = (rows + 7) / 8;
  const int grid = (int)std::min<long long>(std::max<long long>(want, 1), 4096);
  if (d == 64)
    fwd_combine_kernel<64><<<grid, 256, 0, stream>>>(o_part, lse_part, static_cast<uint16_t*>(o), lse, splits, rows);
  else if (d == 256)
    fwd_combine_kernel<256><<<grid, 256, 0, stream>>>(o_part, lse_part, static_cast<uint16_t*>(o), lse, splits, rows);
  else
    fwd_combine_kernel<128><<<grid, 256, 0, stream>>>(o_part, lse_part, static_cast<uint16_t*>(o), lse, splits, rows);
  return cudaGetLastError();
}

// Attention over zero keys: O = 0 and LSE = -inf (the softmax has no term).
__global__ void __launch_bounds__(256) fwd_no_keys_kernel(uint4* __restrict__ o, float* __restrict__ lse, long long n16,
                                                          long long rows) {
  const long long nthr = (long long)gridDim.x * blockDim.x;
  for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < n16; k += nthr) o[k] = make_uint4(0, 0, 0, 0);
  for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < rows; k += nthr) lse[k] = -INFINITY;
}

cudaError_t launch_fwd_no_keys(void* o, float* lse, long long rows, int d, cudaStream_t stream) {
  const long long n16 = rows * d * 2 / 16;
  const long long want = (std::max(n16, rows) + 255) / 256;
  const int grid = (int)std::min<long long>(std::max<long long>(want, 1), 4096);
  fwd_no_keys_kernel<<<grid, 256, 0, stream>>>(static_cast<uint4*>(o), lse, n16, rows);
  return cudaGetLastError();
}

}  // namespace fa
