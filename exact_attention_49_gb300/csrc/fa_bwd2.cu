// fa_bwd2.cu -- the attention backward's main stage on CTA pairs (tcgen05 cta_group::2),
// head dimension 128.
//
// FA4's third co-optimisation (the FA4 summary on ai-papers.net, 提案手法 item 3; the wiki's
// FA4 (3)): tensor memory plus the two-CTA MMA mode, to cut shared-memory traffic and the
// atomic adds of the backward.  A cluster of two CTAs owns 256 consecutive keys of one
// (b, K/V head), 128 per CTA, and walks the same (query head, 128-row query tile) pairs as
// the one-CTA kernel (fa_bwd.cu).  The leader CTA (even rank) issues every MMA for both:
//
//   S^T  = K Q_i^T     M = 256 keys, N = 128 queries   each CTA loads 64 query rows of Q_i
//   dP^T = V dO_i^T    M = 256, N = 128                each CTA loads 64 rows of dO_i
//   dV  += P^T dO_i    M = 256, N = 128 (d), A = P^T from tensor memory;
//                                                      each CTA loads 64 head-dim columns of dO_i
//   dK  += dS^T Q_i    M = 256, N = 128 (d)            each CTA loads 64 columns of Q_i
//   dQ_i^T = K^T dS^T  M = 128 (d), N = 128 queries, K = all 256 keys: the two CTAs' dS^T
//                      halves are exchanged through distributed shared memory, and each CTA
//                      receives dQ^T for its 64 head-dim columns (64 tensor-memory columns)
//
// so every CTA reads half of each B operand from shared memory, and the dQ of a query tile is
// summed over 256 keys on chip before it is added to the fp32 accumulator: half the reduction
// traffic of the one-CTA kernel.  P^T, dS^T and the dQ reductions are computed as in fa_bwd.cu
// (same warps, same arithmetic), each CTA on its own 128 keys.
//
// Warp roles per CTA (448 threads): warps 0-7 compute (P^T, dS^T), warps 8-11 dQ read-out and
// reduction, then the dK/dV epilogue, warp 12 MMA issue (leader only) and tensor-memory
// allocation (both), warp 13 TMA producer.
// Tensor memory per CTA (512 columns, allocated as a pair): dV | dK | S^T (then P^T) |
// dP^T (then dQ^T in its first 64 columns).
// Shared memory per CTA: K, V of its keys; K^T of all 256 keys for its 64 head-dim columns;
// single-buffered halves of Q_i and dO_i (the 64 query rows the S^T / dP^T MMAs need, the 64
// head-dim columns the dK / dV MMAs need); dS^T of its keys; dS^T of all 256 keys for its 64
// query columns (the dQ^T operand, half written by the peer); LSE/D for two query tiles.
#include <algorithm>
#include <type_traits>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

struct Bwd2Cfg {
  static constexpr int D = 128;
  static constexpr int OFF_K = 0;            // own keys [128][128], K-major: chunks d 0-63 | 64-127
  static constexpr int OFF_V = 32768;
  static constexpr int OFF_KQ = 65536;       // [keys of CTA 0 | keys of CTA 1][64 d of this CTA's half]
  static constexpr int OFF_QH = 98304;       // Q rows of this CTA's query half: [64][64] chunks d 0-63 | 64-127
  static constexpr int OFF_QD = 114688;      // Q [128 queries][64 d of this CTA's half]
  static constexpr int OFF_DOH = 131072;     // as QH, for dO
  static constexpr int OFF_DOD = 147456;     // as QD, for dO
  static constexpr int OFF_DS = 163840;      // dS^T own keys [128][128 q]: chunks q 0-63 | 64-127
  static constexpr int OFF_XY = 196608;      // dS^T [keys of CTA 0 | CTA 1][64 q of this CTA's half]
  static constexpr int OFF_LD = 229376;      // two stages of lse2[128] then D[128] (fp32)
  static constexpr int OFF_BAR = 231424;
  static constexpr int NBAR = 20;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static constexpr int THREADS = 448;
  static constexpr uint32_t COL_DV = 0, COL_DK = 128, COL_S = 256, COL_DP = 384;
};
static_assert(Bwd2Cfg::SMEM <= 232448, "shared memory");


__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(448, 1)
    bwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q64,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_do64,
                    const BwdParams p) {
  using C = Bwd2Cfg;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t rank = cluster_rank();
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t kv_full = bar0;
  const uint32_t qh_full = bar0 + 8, qh_empty = bar0 + 16, qd_full = bar0 + 24, qd_empty = bar0 + 32;
  const uint32_t doh_full = bar0 + 40, doh_empty = bar0 + 48, dod_full = bar0 + 56, dod_empty = bar0 + 64;
  auto ld_full = [&](int s) { return bar0 + 72u + 8u * s; };
  auto ld_empty = [&](int s) { return bar0 + 88u + 8u * s; };
  const uint32_t s_full = bar0 + 104, dp_full = bar0 + 112, p_ready = bar0 + 120, ds_ready = bar0 + 128;
  const uint32_t dq_full = bar0 + 136, dq_empty = bar0 + 144, mma_done = bar0 + 152;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const Abort ab{abort, p.status, p.kabort, p.gen};
  // the swizzled layouts need a 1024-byte aligned base; both CTAs see the same base, so both
  // skip all work together (and still meet at the cluster barriers)
  const bool aligned_ok = (sbase & 1023u) == 0;

  // ---- work unit: the cluster's (b, K/V head g, key pair jp); this CTA's key tile j = 2 jp + rank
  const int N = p.Nq;
  const int Np = (N + 127) & ~127;
  const int nq = Np / 128;
  const int BG = p.B * p.Hkv;
  const int nkv = (p.Nk + 127) / 128;
  const int npair = (nkv + 1) / 2;
  constexpr int kHeadGroup = 8;  // CTA order as in fa_bwd.cu: groups of 8 K/V heads, heaviest first
  const int cl = blockIdx.x >> 1;
  const int gi = cl / (kHeadGroup * npair);
  const int gsz = min(kHeadGroup, BG - gi * kHeadGroup);
  const int rem = cl - gi * kHeadGroup * npair;
  const int grp = p.H / p.Hkv;
  // deterministic causal schedules as in fa_bwd.cu, by key pairs
  const bool det_causal = p.deterministic && p.causal;
  const bool desc = det_causal && grp == 1;
  const bool interleave = det_causal && grp > 1;
  const int jp = desc ? npair - 1 - rem / gsz : rem / gsz;
  const int bg = gi * kHeadGroup + rem % gsz;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int j = 2 * jp + (int)rank;
  // causal: the first query tile with a row at or after the pair's first key 256 jp
  const int first = 256 * jp - 127 - p.qoff;
  const int i0 = (p.causal && first > 0) ? (first + 127) / 128 : 0;
  const int ni = max(nq - i0, 0);
  const int ntiles = aligned_ok ? grp * ni : 0;
  auto tile_head = [&](int t) { return b * p.H + g * grp + (interleave ? t % grp : t / ni); };
  auto tile_row = [&](int t) { return interleave ? nq - 1 - t / grp : i0 + t % ni; };

  if (warp == 0 && lane == 0) {
    mbar_init(kv_full, 1);
    mbar_init(qh_full, 1);
    mbar_init(qh_empty, 1);
    mbar_init(qd_full, 1);
    mbar_init(qd_empty, 1);
    mbar_init(doh_full, 1);
    mbar_init(doh_empty, 1);
    mbar_init(dod_full, 1);
    mbar_init(dod_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(ld_full(s), 1);
      mbar_init(ld_empty(s), 8);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 16);   // 8 compute warps in each CTA
    mbar_init(ds_ready, 16);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 8);   // 4 read-out warps in each CTA
    mbar_init(mma_done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  if (warp == 13 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_q64);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_do64);
  }
  if (!aligned_ok && threadIdx.x == 0) atomicCAS(p.status, 0, -5);
  tc_fence_before();
  cluster_sync();  // barrier initialisation visible to the peer before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto lead = [&](uint32_t bar) { return mapa(bar, 0); };  // the leader's copy of a barrier

  if (warp == 13) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0 && ntiles > 0) {
      if (rank == 0) mbar_arrive_expect_tx(kv_full, 2 * 3 * 32768);
      for (int ch = 0; ch < 2; ++ch) {
        tma_load_3d_pair(sbase + C::OFF_K + ch * 16384, &tm_k, lead(kv_full), ch * 64, j * 128, bg);
        tma_load_3d_pair(sbase + C::OFF_V + ch * 16384, &tm_v, lead(kv_full), ch * 64, j * 128, bg);
      }
      for (int blk = 0; blk < 2; ++blk)
        tma_load_3d_pair(sbase + C::OFF_KQ + blk * 16384, &tm_k, lead(kv_full), 64 * (int)rank, (2 * jp + blk) * 128,
                         bg);
      int issued = 0;
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int bh = tile_head(t), i = tile_row(t);
        const int s = t & 1;
        const uint32_t pe = (t & 1) ^ 1;  // single buffers: the previous tile's phase
        // failure-injection test hook (never set in normal use): the leader loads nothing for
        // the second query tile, so the MMA warp's wait on it gives up
        const bool skip = p.debug_hook == 2 && t == 1 && rank == 0;
        if (!mbar_wait_cl(ld_empty(s), ((t >> 1) & 1) ^ 1, ab)) break;
        const size_t row0 = (size_t)bh * Np + (size_t)i * 128;
        mbar_arrive_expect_tx(ld_full(s), 1024);
        bulk_load(sbase + C::OFF_LD + s * 1024, p.lse2 + row0, 512, ld_full(s));
        bulk_load(sbase + C::OFF_LD + s * 1024 + 512, p.dvec + row0, 512, ld_full(s));
        ok = mbar_wait_cl(qh_empty, pe, ab);
        if (ok && !skip) {
          if (rank == 0) mbar_arrive_expect_tx(qh_full, 2 * 16384);
          for (int ch = 0; ch < 2; ++ch)
            tma_load_3d_pair(sbase + C::OFF_QH + ch * 8192, &tm_q64, lead(qh_full), ch * 64, i * 128 + 64 * (int)rank, bh);
        }
        ok = ok && mbar_wait_cl(doh_empty, pe, ab);
        if (ok && !skip) {
          if (rank == 0) mbar_arrive_expect_tx(doh_full, 2 * 16384);
          for (int ch = 0; ch < 2; ++ch)
            tma_load_3d_pair(sbase + C::OFF_DOH + ch * 8192, &tm_do64, lead(doh_full), ch * 64, i * 128 + 64 * (int)rank,
                             bh);
        }
        ok = ok && mbar_wait_cl(dod_empty, pe, ab);
        if (ok && !skip) {
          if (rank == 0) mbar_arrive_expect_tx(dod_full, 2 * 16384);
          tma_load_3d_pair(sbase + C::OFF_DOD, &tm_do, lead(dod_full), 64 * (int)rank, i * 128, bh);
        }
        ok = ok && mbar_wait_cl(qd_empty, pe, ab);
        if (ok && !skip) {
          if (rank == 0) mbar_arrive_expect_tx(qd_full, 2 * 16384);
          tma_load_3d_pair(sbase + C::OFF_QD, &tm_q, lead(qd_full), 64 * (int)rank, i * 128, bh);
        }
        if (ok) issued = t + 1;
      }
      if (*abort) {
        // The pair gave up.  The leader waits (bounded) for the phases it armed, which also
        // complete when the peer's copies land; then both wait a short grace period so that
        // no copy is in flight when the cluster exits.
        auto drain = [&](uint32_t bar, uint32_t parity) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait_cl(bar, parity) && globaltimer() - t0 < 1000000ull) {
          }
        };
        for (int t = max(0, issued - 2); t < issued; ++t) drain(ld_full(t & 1), (t >> 1) & 1);
        if (rank == 0) {
          drain(kv_full, 0);
          if (issued > 0) {
            const uint32_t last = (issued - 1) & 1;
            drain(qh_full, last);
            drain(doh_full, last);
            drain(dod_full, last);
            drain(qd_full, last);
          }
        }
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 50000ull) {
        }
      }
    }
  } else if (warp == 12) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (rank == 0 && lane == 0 && ntiles > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(256, 128, false, false);  // S^T, dP^T
      constexpr uint32_t idKV = idesc_bf16_f32(256, 128, false, true);  // dV, dK (B: MN-major)
      constexpr uint32_t idQ = idesc_bf16_f32(128, 128, true, true);    // dQ^T (A, B: MN-major)
      const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sKQ = sbase + C::OFF_KQ;
      const uint32_t sQH = sbase + C::OFF_QH, sQD = sbase + C::OFF_QD;
      const uint32_t sDOH = sbase + C::OFF_DOH, sDOD = sbase + C::OFF_DOD;
      const uint32_t sDS = sbase + C::OFF_DS, sXY = sbase + C::OFF_XY;
      // D[256 keys x 128 queries] = A[keys][d] . B[64 queries per CTA][d]^T, both K-major
      auto ss_kmajor = [&](uint32_t dcol, uint32_t a, uint32_t bsm) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_pair(tmem + dcol, sdesc_sw128(a + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(bsm + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), idS, kk > 0);
      };
      bool ok = mbar_wait_cl(kv_full, 0, ab) && mbar_wait_cl(qh_full, 0, ab);
      if (ok) {
        tc_fence_after();
        ss_kmajor(C::COL_S, sK, sQH);
        mma_commit_pair(s_full);
        mma_commit_pair(qh_empty);
        ok = mbar_wait_cl(doh_full, 0, ab);
      }
      if (ok) {
        tc_fence_after();
        ss_kmajor(C::COL_DP, sV, sDOH);
        mma_commit_pair(dp_full);
        mma_commit_pair(doh_empty);
      }
      auto step = [&](int t, auto more_tiles) -> bool {
        constexpr bool MORE = decltype(more_tiles)::value;
        const uint32_t par = t & 1, npar = (t + 1) & 1;
        if (!mbar_wait_cl(p_ready, par, ab) || !mbar_wait_cl(dod_full, par, ab)) return false;
        tc_fence_after();
        // dV += P^T dO_t: A = P^T from tensor memory (queries 0-63 in columns 0-31, 64-127 in
        // 64-95 of the S^T block), B = this CTA's 64 head-dim columns of dO_t
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_pair(tmem + C::COL_DV, tmem + C::COL_S + 64 * (kk >> 2) + (kk & 3) * 8,
                      sdesc_sw128(sDOD + kk * 2048, 16384, 1024), idKV, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit_pair(dod_empty);
        if constexpr (MORE) {
          if (!mbar_wait_cl(qh_full, npar, ab)) return false;
          tc_fence_after();
          ss_kmajor(C::COL_S, sK, sQH);  // S^T of the next tile (P^T_t already consumed)
          mma_commit_pair(s_full);
          mma_commit_pair(qh_empty);
        }
        if (!mbar_wait_cl(ds_ready, par, ab)) return false;
        tc_fence_after();
        // dQ_t^T = K^T dS^T over all 256 keys (16 steps of 16 keys: this CTA's keys, then the
        // peer's), into the first 64 columns of the dP^T block
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          mma_ss_pair(tmem + C::COL_DP, sdesc_sw128(sKQ + (kk >> 3) * 16384 + (kk & 7) * 2048, 16384, 1024),
                      sdesc_sw128(sXY + (kk >> 3) * 16384 + (kk & 7) * 2048, 16384, 1024), idQ, kk > 0);
        mma_commit_pair(dq_full);
        if (!mbar_wait_cl(qd_full, par, ab)) return false;
        tc_fence_after();
        // dK += dS^T Q_t: A = dS^T of this CTA's keys (K-major over queries), B = this CTA's 64
        // head-dim columns of Q_t
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_pair(tmem + C::COL_DK, sdesc_sw128(sDS + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(sQD + kk * 2048, 16384, 1024), idKV, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit_pair(qd_empty);
        if constexpr (MORE) {
          if (!mbar_wait_cl(dq_empty, par, ab) || !mbar_wait_cl(doh_full, npar, ab)) return false;
          tc_fence_after();
          ss_kmajor(C::COL_DP, sV, sDOH);
          mma_commit_pair(dp_full);
          mma_commit_pair(doh_empty);
        }
        return true;
      };
      for (int t = 0; ok && t + 1 < ntiles; ++t) ok = step(t, std::true_type{});
      if (ok) ok = step(ntiles - 1, std::false_type{});
      // every MMA of the pair has completed when mma_done fires in both CTAs
      mma_commit_pair(mma_done);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute: P^T and dS^T
    const int w = warp >> 2;           // query-column half
    const int r = threadIdx.x & 127;   // key row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::COL_S + 64 * w;
    const uint32_t tDP = tmem + lane_off + C::COL_DP + 64 * w;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t scx2 = f2_pack(p.scale, p.scale);
    uint8_t* ds_row = smem + C::OFF_DS + w * 16384 + r * 128;
    // the dQ^T operand: dS^T of this CTA's keys for query half w goes to block `rank` of the
    // XY buffer of the CTA that owns query half w (this CTA when w == rank, else the peer)
    const uint32_t xy_row = mapa(sbase + C::OFF_XY + rank * 16384 + r * 128, (uint32_t)w);
    const bool key_pad = j * 128 + r >= p.Nk;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t & 1;
      const int cut = p.causal ? r + 128 * (j - tile_row(t)) - 64 * w - p.qoff : 0;
      const float4* lse4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 1024) + 16 * w;
      const float4* d4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 1024 + 512) + 16 * w;
      if (!__all_sync(0xffffffffu, mbar_wait_cl(ld_full(s), (t >> 1) & 1, ab))) break;
      if (!__all_sync(0xffffffffu, mbar_wait_cl(s_full, t & 1, ab))) break;
      tc_fence_after();
      float pv[64];
      {
        uint32_t ra[32], rb[32];
        tmem_ld32_nowait(tS, ra);
        tmem_wait_ld(ra);
        tmem_ld32_nowait(tS + 32, rb);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          if (c4 == 8) tmem_wait_ld(rb);
          const float4 L = lse4[c4];
          const uint32_t* src = (c4 < 8) ? ra : rb;
          const int o = (c4 & 7) * 4;
          const float2 x01 = f2_unpack(f2_fma(f2_pack(__uint_as_float(src[o]), __uint_as_float(src[o + 1])), sl2x2,
                                              f2_pack(-L.x, -L.y)));
          const float2 x23 = f2_unpack(f2_fma(f2_pack(__uint_as_float(src[o + 2]), __uint_as_float(src[o + 3])), sl2x2,
                                              f2_pack(-L.z, -L.w)));
          pv[4 * c4] = ex2_mufu(x01.x);
          pv[4 * c4 + 1] = ex2_mufu(x01.y);
          pv[4 * c4 + 2] = ex2_mufu(x23.x);
          pv[4 * c4 + 3] = ex2_mufu(x23.y);
        }
      }
      if (key_pad) {
#pragma unroll
        for (int c = 0; c < 64; ++c) pv[c] = 0.f;
      }
      if (cut > 0) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < cut) pv[c] = 0.f;
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) pk[c2] = pack_bf16x2(pv[32 * cc + 2 * c2], pv[32 * cc + 2 * c2 + 1]);
        tmem_st16(tS + 16 * cc, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lead(p_ready));

      if (!__all_sync(0xffffffffu, mbar_wait_cl(dp_full, t & 1, ab))) break;
      tc_fence_after();
      {
        uint32_t ra[32], rb[32];
        tmem_ld32_nowait(tDP, ra);
        tmem_wait_ld(ra);
        tmem_ld32_nowait(tDP + 32, rb);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          if (cc == 1) tmem_wait_ld(rb);
          const uint32_t* src = cc ? rb : ra;
          uint32_t pk[16];
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 Dv = d4[8 * cc + c4];
            const int o = 4 * c4, q = 32 * cc + 4 * c4;
            const uint64_t a = f2_add(f2_pack(__uint_as_float(src[o]), __uint_as_float(src[o + 1])), f2_pack(-Dv.x, -Dv.y));
            const uint64_t bb = f2_add(f2_pack(__uint_as_float(src[o + 2]), __uint_as_float(src[o + 3])),
                                       f2_pack(-Dv.z, -Dv.w));
            const float2 d01 = f2_unpack(f2_mul(f2_mul(a, f2_pack(pv[q], pv[q + 1])), scx2));
            const float2 d23 = f2_unpack(f2_mul(f2_mul(bb, f2_pack(pv[q + 2], pv[q + 3])), scx2));
            pk[2 * c4] = pack_bf16x2(d01.x, d01.y);
            pk[2 * c4 + 1] = pack_bf16x2(d23.x, d23.y);
          }
          // dS^T row r, queries [32cc, 32cc+32) of this half: four 16-byte pieces, 128B-swizzled,
          // into this CTA's dS^T tile and into the dQ^T operand (here or in the peer)
#pragma unroll
          for (int pc = 0; pc < 4; ++pc) {
            const int piece = 4 * cc + pc;
            const uint4 v = make_uint4(pk[4 * pc], pk[4 * pc + 1], pk[4 * pc + 2], pk[4 * pc + 3]);
            const uint32_t off = (uint32_t)((piece ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(ds_row + off) = v;
            st_cluster_v4(xy_row + off, v);
          }
        }
      }
      fence_async_smem_cluster();  // dS^T visible to the MMAs (async proxy), here and in the peer
      tc_fence_before();           // TMEM loads of dP^T done before the dQ^T MMA overwrites it
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(lead(ds_ready));
        mbar_arrive(ld_empty(s));
      }
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ read-out, dK/dV epilogue
    // dQ^T of this CTA's 64 head-dim columns: TMEM lane L holds column 64 rank + (L % 64) for
    // queries 64 (L / 64) + c, c = 0..63 (tensor-memory columns of the dP^T block)
    const int L = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDQ = tmem + lane_off + C::COL_DP;
    const int dcol = 64 * (int)rank + (L & 63);
    const int qbase = (L >> 6) * 64;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int bh = tile_head(t), i = tile_row(t);
      ok = __all_sync(0xffffffffu, mbar_wait_cl(dq_full, t & 1, ab));
      if (!ok) break;
      tc_fence_after();
      int* counter = p.deterministic ? p.counters + ((size_t)bh * nq + i) : nullptr;
      // this pair's place in the fixed order of query tile i's contributions (as in fa_bwd.cu,
      // by key pairs): both CTAs of each earlier pair add their halves before this pair starts
      const int rank_p = desc ? min(npair - 1, (128 * i + 127 + p.qoff) / 256) - jp : jp;
      if (p.deterministic) {
        if (L == 0) {
          const uint64_t t0 = globaltimer();
          while (ld_acquire(counter) < 2 * rank_p) {
            const unsigned long long el = globaltimer() - t0;
            if (should_stop(ab, el)) break;
            if (el > kWaitLimitNs) {
              give_up(ab);
              break;
            }
          }
        }
        named_bar(1, 128);
      }
      uint32_t va[32], vb[32];
      tmem_ld32_nowait(tDQ, va);
      tmem_ld32_nowait(tDQ + 32, vb);
      tmem_wait_ld(va);
      tmem_wait_ld(vb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lead(dq_empty));
      // a warp adds 32 consecutive head-dim columns of one query row per instruction (128 bytes);
      // in deterministic mode only this pair adds to query tile i now, so the order is fixed
      if (!p.deterministic || !*abort) {
        float* col = p.dq_acc + ((size_t)bh * Np + (size_t)i * 128 + qbase) * D + dcol;
#pragma unroll
        for (int m = 0; m < 32; ++m) red_add(col + (size_t)m * D, __uint_as_float(va[m]));
#pragma unroll
        for (int m = 0; m < 32; ++m) red_add(col + (size_t)(32 + m) * D, __uint_as_float(vb[m]));
      }
      if (p.deterministic) {
        __threadfence();
        named_bar(1, 128);
        // (failure-injection test hook: the first pair keeps its successors waiting)
        if (L == 0 && !(p.debug_hook == 1 && cl == 0)) red_add_release(counter, 1);
      }
    }
    // mma_done fires after every MMA of the pair, the last dK one included
    if (ok && ntiles > 0) ok = __all_sync(0xffffffffu, mbar_wait_cl(mma_done, 0, ab));
    if (ok) {
      tc_fence_after();
      const size_t krow = (size_t)bg * p.Nk + (size_t)j * 128 + L;
      const bool krow_valid = j * 128 + L < p.Nk;  // the last key tile may run past Nk
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(which ? p.dk : p.dv) + krow * D);
        const uint32_t tcol = tmem + lane_off + (which ? C::COL_DK : C::COL_DV);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tcol + 32 * c, v);
          if (ntiles == 0) {  // no query row sees these keys: their gradients are zero
#pragma unroll
            for (int m = 0; m < 32; ++m) v[m] = 0u;
          }
#pragma unroll
          for (int m = 0; m < 4; ++m)
            if (krow_valid)
              out[4 * c + m] =
                  make_uint4(pack_bf16x2(__uint_as_float(v[8 * m]), __uint_as_float(v[8 * m + 1])),
                             pack_bf16x2(__uint_as_float(v[8 * m + 2]), __uint_as_float(v[8 * m + 3])),
                             pack_bf16x2(__uint_as_float(v[8 * m + 4]), __uint_as_float(v[8 * m + 5])),
                             pack_bf16x2(__uint_as_float(v[8 * m + 6]), __uint_as_float(v[8 * m + 7])));
        }
      }
    }
  }

  // Neither CTA leaves while the pair's MMAs, copies or remote arrivals may still touch its
  // memory: the leader's MMA warp waits (bounded, even after an abort) for its last commit,
  // then both meet at the cluster barrier and free the paired tensor memory.
  if (warp == 12 && rank == 0 && lane == 0 && ntiles > 0) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait_cl(mma_done, 0) && globaltimer() - t0 < kWaitLimitNs) {
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

cudaError_t launch_bwd_main_pair(const CUtensorMap& tq, const CUtensorMap& tq64, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdo64,
                                 const BwdParams& p, cudaStream_t stream) {
  using C = Bwd2Cfg;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(bwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int nkv = (p.Nk + 127) / 128;
  const long long blocks = 2LL * ((nkv + 1) / 2) * p.B * p.Hkv;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  bwd_pair_kernel<<<dim3((unsigned)blocks), dim3(C::THREADS), C::SMEM, stream>>>(tq, tq64, tk, tv, tdo, tdo64, p);
  return cudaGetLastError();
}

}  // namespace fa
