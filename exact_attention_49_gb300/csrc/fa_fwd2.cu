// fa_fwd2.cu -- the attention forward on CTA pairs (tcgen05 cta_group::2), head dimension 128.
//
// The same method as fa_fwd.cu (tiling and online softmax with conditional rescale: the
// explainer's tiling and online-softmax paragraphs; FA4's conditional rescale, ai-papers.net
// summary 提案手法 item 2), with FA4's larger MMA tiles (提案手法 item 1; wiki FA4 (1)): a
// cluster of two CTAs runs M = 256 MMAs over 512 query rows of one head.
//
//   S_w  = Q_w K_j^T    M = 256 (128 rows of each CTA), N = 128 keys: each CTA loads 64 of
//                       the tile's keys, all head-dimension columns
//   O_w += P_w V_j      M = 256, N = 128 (d): each CTA loads all 128 keys of V_j for its 64
//                       head-dimension columns
//
// With the K/V ring slots halved, shared memory holds P as well: the softmax warps write the
// bf16 probabilities to shared memory instead of over S in tensor memory, so the MMA warp can
// compute S_w of the next key tile as soon as the softmax warps have read S_w of this one,
// while they are still computing exponentials (in fa_fwd.cu, P overwrites S, and the next S
// waits for this tile's PV).  Per CTA: query tile w (w = 0, 1) covers rows q0 + 256 w + 128 rank
// of the unit's 512; its softmax warpgroup w works on its own rows only.
//
// Warp roles per CTA (384 threads, setmaxnreg split as in fa_fwd.cu): warps 0-3 softmax of
// query tile 0, warps 4-7 of query tile 1, warp 8 MMA issue (leader only) and tensor-memory
// allocation (both), warp 9 TMA producer, warps 10-11 idle.
// Tensor memory per CTA (512 columns, allocated as a pair): S0 | S1 | O0 | O1.
// Shared memory per CTA: Q0, Q1 (own rows), P0, P1, a ring of six 16 KB slots holding K and V
// halves in turn.
#include <algorithm>
#include <type_traits>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

struct Fwd2Cfg {
  static constexpr int D = 128;
  static constexpr int TILE = 32768;         // 128 x 128 bf16
  static constexpr int SLOT = 16384;         // a K half [64 keys][128 d] or a V half [128 keys][64 d]
  static constexpr int STAGES = 6;
  static constexpr int OFF_Q = 0;            // Q0 | Q1, each [128 rows][128 d], chunks d 0-63 | 64-127
  static constexpr int OFF_P = 2 * TILE;     // P0 | P1, each [128 rows][128 keys], chunks keys 0-63 | 64-127
  static constexpr int OFF_RING = 4 * TILE;
  static constexpr int OFF_BAR = OFF_RING + STAGES * SLOT;
  static constexpr int NBAR = 2 * STAGES + 13;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr int THREADS = 384;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 384;
  static constexpr int REG_SOFTMAX = 184, REG_OTHER = 136;  // of 168 at launch (see fa_fwd.cu)
};
static_assert(Fwd2Cfg::SMEM_BYTES <= 232448, "shared memory");

struct Fwd2Unit {
  int bh, q0, kv_z;
  int n0, n1;  // key tiles seen by the rows of query tile 0 (rows q0..q0+255) and tile 1
  bool two;    // the unit has rows in query tile 1 (rows q0+256..q0+511)
};

// Units: blocks of 512 query rows of one (b, h), heaviest first under a causal mask.
FA_DEV Fwd2Unit fwd2_unit(const FwdParams& p, int u) {
  const int N = p.Nq;
  const int ncb = (N + 511) / 512;
  const int BH = p.B * p.H;
  Fwd2Unit w;
  const int cb = p.causal ? (ncb - 1 - u / BH) : (u / BH);
  w.bh = u % BH;
  const int b = w.bh / p.H, h = w.bh % p.H;
  w.kv_z = b * p.Hkv + h / (p.H / p.Hkv);
  w.q0 = cb * 512;
  const int n_kv_all = (p.Nk + 127) / 128;
  auto visible = [&](int last_row) {  // key tiles a block whose last row is last_row needs
    const int k_last = last_row + p.qoff;
    return p.causal ? (k_last < 0 ? 1 : min(n_kv_all, k_last / 128 + 1)) : n_kv_all;
  };
  w.two = N - w.q0 > 256;
  w.n0 = visible(min(w.q0 + 255, N - 1));
  w.n1 = w.two ? visible(min(w.q0 + 511, N - 1)) : w.n0;
  return w;
}

FA_DEV int fwd2_unit_index(int r) {  // boustrophedon order over clusters (see fa_fwd.cu)
  const int G = gridDim.x >> 1, c = blockIdx.x >> 1;
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
    fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k64,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p, int n_units) {
  using C = Fwd2Cfg;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rank = cluster_rank();
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  const uint32_t q_full = bar0 + 8u * (2 * C::STAGES), q_empty = bar0 + 8u * (2 * C::STAGES + 1);
  auto s_full = [&](int w) { return bar0 + 8u * (2 * C::STAGES + 2 + w); };
  auto s_free = [&](int w) { return bar0 + 8u * (2 * C::STAGES + 4 + w); };
  auto p_full = [&](int w) { return bar0 + 8u * (2 * C::STAGES + 6 + w); };
  auto o_bar = [&](int w) { return bar0 + 8u * (2 * C::STAGES + 8 + w); };
  auto o_free = [&](int w) { return bar0 + 8u * (2 * C::STAGES + 10 + w); };
  const uint32_t mma_done = bar0 + 8u * (2 * C::STAGES + 12);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const Abort ab{abort, p.status, p.kabort, p.gen};
  const int warp = warp_id();
  const int lane = lane_id();
  const int N = p.Nq;
  auto lead = [&](uint32_t bar) { return mapa(bar, 0); };

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int w = 0; w < 2; ++w) {
      mbar_init(s_full(w), 1);
      mbar_init(s_free(w), 8);  // 4 softmax warps in each CTA
      mbar_init(p_full(w), 8);
      mbar_init(o_bar(w), 1);
      mbar_init(o_free(w), 8);
    }
    mbar_init(mma_done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  if (warp == 9 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k64);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  cluster_sync();  // barrier initialisation visible to the peer before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_OTHER));
    if (warp == 9 && lane == 0) {
      // ---------------------------------------------------------- TMA producer (both CTAs)
      uint32_t it = 0, issued = 0, q_loads = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int u = fwd2_unit_index(r);
        if (u >= n_units) break;
        const Fwd2Unit w = fwd2_unit(p, u);
        if (q_loads > 0 && !mbar_wait_cl(q_empty, (q_loads - 1) & 1, ab)) break;
        if (rank == 0) mbar_arrive_expect_tx(q_full, (w.two ? 2 : 1) * 2 * C::TILE);
        for (int qt = 0; qt < (w.two ? 2 : 1); ++qt)
          for (int ch = 0; ch < 2; ++ch)
            tma_load_3d_pair(sbase + C::OFF_Q + qt * C::TILE + ch * 16384, &tm_q, lead(q_full), ch * 64,
                             w.q0 + 256 * qt + 128 * (int)rank, w.bh);
        ++q_loads;
        for (int jj = 0; jj < 2 * w.n1; ++jj, ++it) {
          const uint32_t slot = it % C::STAGES;
          // failure-injection test hook (never set in normal use): the leader skips one load
          if (r == 0 && jj == p.drop_it && rank == 0) continue;
          if (!mbar_wait_cl(empty_bar(slot), ((it / C::STAGES) & 1) ^ 1, ab)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(full_bar(slot), 2 * C::SLOT);
          const int j = jj >> 1;
          const uint32_t dst = sbase + C::OFF_RING + slot * C::SLOT;
          if ((jj & 1) == 0) {  // K: this CTA's 64 keys of the tile, both head-dimension chunks
            for (int ch = 0; ch < 2; ++ch)
              tma_load_3d_pair(dst + ch * 8192, &tm_k64, lead(full_bar(slot)), ch * 64, j * 128 + 64 * (int)rank,
                               w.kv_z);
          } else {  // V: all 128 keys of the tile, this CTA's 64 head-dimension columns
            tma_load_3d_pair(dst, &tm_v, lead(full_bar(slot)), 64 * (int)rank, j * 128, w.kv_z);
          }
          issued = it + 1;
        }
      }
      if (*abort) {
        // the pair gave up: the leader waits (bounded) for the phases it armed, which also
        // complete when the peer's copies land; both then wait a short grace period
        auto drain = [&](uint32_t bar, uint32_t parity) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait_cl(bar, parity) && globaltimer() - t0 < 1000000ull) {
          }
        };
        if (rank == 0) {
          for (uint32_t k = issued > C::STAGES ? issued - C::STAGES : 0; k < issued; ++k)
            drain(full_bar(k % C::STAGES), (k / C::STAGES) & 1);
          if (q_loads > 0) drain(q_full, (q_loads - 1) & 1);
        }
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 50000ull) {
        }
      }
    } else if (warp == 8 && lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer (leader)
      constexpr uint32_t idS = idesc_bf16_f32(256, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(256, 128, false, true);
      auto slot_of = [](uint32_t k) { return k % C::STAGES; };
      auto par_of = [](uint32_t k) { return (k / C::STAGES) & 1u; };
      // S_w = Q_w K^T: A = this CTA's query rows, B = its 64 keys of the tile (K-major)
      auto issue_s = [&](int w, uint32_t slot) {
        const uint32_t a0 = sbase + C::OFF_Q + w * C::TILE, b0 = sbase + C::OFF_RING + slot * C::SLOT;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_pair(tmem + (w ? C::COL_S1 : C::COL_S0),
                      sdesc_sw128(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(b0 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), idS, kk > 0);
      };
      // O_w += P_w V: A = P_w (K-major over keys) in shared memory, B = this CTA's 64
      // head-dimension columns of V (MN-major)
      auto issue_pv = [&](int w, uint32_t slot, bool acc) {
        const uint32_t a0 = sbase + C::OFF_P + w * C::TILE, b0 = sbase + C::OFF_RING + slot * C::SLOT;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_pair(tmem + (w ? C::COL_O1 : C::COL_O0),
                      sdesc_sw128(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(b0 + kk * 2048, 16384, 1024), idO, (acc || kk > 0) ? 1u : 0u);
      };
      uint32_t it = 0, units = 0, units2 = 0, jg0 = 0, jg1 = 0;
      // One step of a unit: PV of key tile j for the active query tiles, preceded by S of key
      // tile j + 1 (NEXT0 / NEXT1) as soon as the softmax warps have read S of tile j.
      auto step = [&](int j, auto has0, auto has1, auto next0, auto next1, uint32_t it0, uint32_t g0, uint32_t g1,
                      int last_s) -> bool {
        constexpr bool H0 = decltype(has0)::value, H1 = decltype(has1)::value;
        constexpr bool X0 = decltype(next0)::value, X1 = decltype(next1)::value;
        const uint32_t itv = it0 + 2 * j + 1, itk = itv + 1;
        if constexpr (X0 || X1) {
          if (!mbar_wait_cl(full_bar(slot_of(itk)), par_of(itk), ab)) return false;
          if constexpr (X0) {
            if (!mbar_wait_cl(s_free(0), (g0 + j) & 1, ab)) return false;
            tc_fence_after();
            issue_s(0, slot_of(itk));
            mma_commit_pair(s_full(0));
          }
          if constexpr (X1) {
            if (!mbar_wait_cl(s_free(1), (g1 + j) & 1, ab)) return false;
            tc_fence_after();
            issue_s(1, slot_of(itk));
            mma_commit_pair(s_full(1));
          }
          if (j + 1 == last_s) mma_commit_pair(q_empty);  // the unit's last S MMAs
          mma_commit_pair(empty_bar(slot_of(itk)));
        }
        if (!mbar_wait_cl(full_bar(slot_of(itv)), par_of(itv), ab)) return false;
        if constexpr (H0) {
          if (!mbar_wait_cl(p_full(0), (g0 + j) & 1, ab)) return false;
          tc_fence_after();
          issue_pv(0, slot_of(itv), j > 0);
          mma_commit_pair(o_bar(0));
        }
        if constexpr (H1) {
          if (!mbar_wait_cl(p_full(1), (g1 + j) & 1, ab)) return false;
          tc_fence_after();
          issue_pv(1, slot_of(itv), j > 0);
          mma_commit_pair(o_bar(1));
        }
        mma_commit_pair(empty_bar(slot_of(itv)));
        return true;
      };
      using T = std::true_type;
      using F = std::false_type;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int u = fwd2_unit_index(r);
        if (u >= n_units) break;
        const Fwd2Unit w = fwd2_unit(p, u);
        const int n0 = w.n0, n1 = w.n1;
        const int last_s = w.two ? n1 - 1 : n0 - 1;
        ok = mbar_wait_cl(q_full, units & 1, ab) && mbar_wait_cl(full_bar(slot_of(it)), par_of(it), ab);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, slot_of(it));
        mma_commit_pair(s_full(0));
        if (w.two) {
          issue_s(1, slot_of(it));
          mma_commit_pair(s_full(1));
        }
        if (last_s == 0) mma_commit_pair(q_empty);
        mma_commit_pair(empty_bar(slot_of(it)));
        // the first PV of a query tile overwrites its O accumulator: wait until the previous
        // unit's epilogue has read it out (its softmax warps release it before they start here)
        if (units > 0) ok = mbar_wait_cl(o_free(0), (units - 1) & 1, ab);
        if (ok && w.two && units2 > 0) ok = mbar_wait_cl(o_free(1), (units2 - 1) & 1, ab);
        if (w.two) {
          // j < n0 - 1: both tiles, both next S; j = n0 - 1: tile 0's last; then tile 1 alone
          for (int j = 0; ok && j + 1 < n0; ++j) ok = step(j, T{}, T{}, T{}, T{}, it, jg0, jg1, last_s);
          if (ok) {
            if (n1 > n0)
              ok = step(n0 - 1, T{}, T{}, F{}, T{}, it, jg0, jg1, last_s);
            else
              ok = step(n0 - 1, T{}, T{}, F{}, F{}, it, jg0, jg1, last_s);
          }
          for (int j = n0; ok && j + 1 < n1; ++j) ok = step(j, F{}, T{}, F{}, T{}, it, jg0, jg1, last_s);
          if (ok && n1 > n0) ok = step(n1 - 1, F{}, T{}, F{}, F{}, it, jg0, jg1, last_s);
        } else {
          for (int j = 0; ok && j + 1 < n0; ++j) ok = step(j, T{}, F{}, T{}, F{}, it, jg0, jg1, last_s);
          if (ok) ok = step(n0 - 1, T{}, F{}, F{}, F{}, it, jg0, jg1, last_s);
        }
        it += 2 * w.n1;
        jg0 += n0;
        ++units;
        if (w.two) {
          jg1 += n1;
          ++units2;
        }
      }
      mma_commit_pair(mma_done);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_SOFTMAX));
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int w = warp >> 2;            // query tile
    const int r = threadIdx.x & 127;    // row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (w ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = tmem + lane_off + (w ? C::COL_O1 : C::COL_O0);
    uint8_t* p_row = smem + C::OFF_P + w * C::TILE + r * 128;  // row r of P_w, chunk 0 (chunk 1: +16 KB)
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    int jg = 0;  // key tiles processed by this warpgroup (s_full, o_bar phases)
    bool ok = true;
    for (int ru = 0; ok; ++ru) {
      const int u = fwd2_unit_index(ru);
      if (u >= n_units) break;
      const Fwd2Unit wu = fwd2_unit(p, u);
      if (w == 1 && !wu.two) continue;
      const int n_kv = w ? wu.n1 : wu.n0;
      const int tile_row0 = wu.q0 + 256 * w + 128 * (int)rank;
      const int row = tile_row0 + r;
      float m_used = -INFINITY;
      uint64_t l_exact = 0;
      float lr0 = 0.f, lr1 = 0.f;  // sum of the bf16 weights (see fa_fwd.cu)
      bool o_ready = false;        // this tile's previous PV known complete
      for (int j = 0; j < n_kv; ++j, ++jg) {
        ok = __all_sync(0xffffffffu, mbar_wait_cl(s_full(w), jg & 1, ab));
        if (!ok) break;
        tc_fence_after();
        float s[128];
        {
          uint32_t rr[128];
          tmem_ld128(tS, rr);
#pragma unroll
          for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(rr[i]);
        }
        // S_w has been read: the MMA warp may compute the next key tile's S into it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead(s_free(w)));
        o_ready = false;
        const int col0 = j * 128;
        if ((p.causal && col0 + 127 > tile_row0 + p.qoff) || col0 + 128 > p.Nk) {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int col = col0 + c;
            if ((p.causal && col > row + p.qoff) || col >= p.Nk) s[c] = -INFINITY;
          }
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
            if (p.rescale_events) {
              const unsigned moved = __ballot_sync(0xffffffffu, alpha != 1.f);
              if (lane == 0) atomicAdd(p.rescale_events, (unsigned long long)__popc(moved));
            }
            ok = __all_sync(0xffffffffu, mbar_wait_cl(o_bar(w), (jg - 1) & 1, ab));
            if (!ok) break;
            o_ready = true;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
              uint32_t rr[16];
              tmem_ld16(tO + 16 * c, rr);
#pragma unroll
              for (int i = 0; i < 16; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
              tmem_st16(tO + 16 * c, rr);
            }
            tmem_st_wait();
          }
          l_exact = f2_mul(l_exact, f2_pack(alpha, alpha));
          lr0 *= alpha;
          lr1 *= alpha;
          m_used = m_new;
        }
        const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
        const uint64_t nm2 = f2_pack(neg_m, neg_m);
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float2 x = f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sl2x2, nm2));
          const float p0 = ex2_mufu(x.x), p1 = ex2_mufu(x.y);
          pk[i] = pack_bf16x2(p0, p1);
          l_exact = f2_add(l_exact, f2_pack(p0, p1));
          if (i & 1)
            lr1 = add_bf16_hi(add_bf16_lo(lr1, pk[i]), pk[i]);
          else
            lr0 = add_bf16_hi(add_bf16_lo(lr0, pk[i]), pk[i]);
        }
        // P_w is free once the previous key tile's PV has completed
        if (jg > 0 && !o_ready) {
          ok = __all_sync(0xffffffffu, mbar_wait_cl(o_bar(w), (jg - 1) & 1, ab));
          if (!ok) break;
        }
        // row r of P_w: keys 0-63 in chunk 0, 64-127 in chunk 1, 16-byte pieces 128B-swizzled
#pragma unroll
        for (int piece = 0; piece < 16; ++piece) {
          uint8_t* dst = p_row + (piece >> 3) * 16384 + (((piece & 7) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) =
              make_uint4(pk[4 * piece], pk[4 * piece + 1], pk[4 * piece + 2], pk[4 * piece + 3]);
        }
        fence_async_smem();  // P visible to the MMAs (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead(p_full(w)));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> bf16, LSE = ln 2 * (m_used + log2 l); O's tensor memory is
      // handed back right after the last load from it
      ok = __all_sync(0xffffffffu, mbar_wait_cl(o_bar(w), (jg - 1) & 1, ab));
      if (!ok) break;
      tc_fence_after();
      const float2 le = f2_unpack(l_exact);
      const float l = le.x + le.y, lrs = lr0 + lr1;
      const float inv_l = lrs > 0.f ? 1.f / lrs : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + ((size_t)wu.bh * N + row) * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tO + 32 * c, rr);
        if (c == D / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lead(o_free(w)));
        }
        uint32_t pko[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pko[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * inv_l, __uint_as_float(rr[2 * i + 1]) * inv_l);
        if (row < N) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            orow[c * 4 + v4] = make_uint4(pko[4 * v4], pko[4 * v4 + 1], pko[4 * v4 + 2], pko[4 * v4 + 3]);
        }
      }
      if (row < N) p.lse[(size_t)wu.bh * N + row] = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  // Neither CTA leaves while the pair's MMAs or copies may still touch its memory.
  if (warp == 8 && lane == 0 && rank == 0) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait_cl(mma_done, 0) && globaltimer() - t0 < kWaitLimitNs) {
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

static int fwd2_sm_count() {
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

cudaError_t launch_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tk64, const CUtensorMap& tv, const FwdParams& p,
                            cudaStream_t stream) {
  using C = Fwd2Cfg;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(fwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const long long units = (long long)((p.Nq + 511) / 512) * p.B * p.H;
  if (units > 0x3fffffffLL) return cudaErrorInvalidValue;
  // persistent: one cluster per pair of SMs (at most one per unit)
  const int clusters = (int)std::min<long long>(units, fwd2_sm_count() / 2);
  fwd_pair_kernel<<<dim3((unsigned)(2 * clusters)), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(tq, tk64, tv, p,
                                                                                                (int)units);
  return cudaGetLastError();
}

}  // namespace fa
