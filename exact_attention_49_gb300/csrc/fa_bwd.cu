// fa_bwd.cu -- exact attention backward for sm_103a.
//
// The backward recomputes P from the LSE saved by the forward instead of
// storing it ("FlashAttention" wiki note, 定義 item (2); the explainer's
// recomputation paragraph).  Three kernels:
//
//   preprocess   per query row: D = sum_c dO_c O_c (fp32) and LSE in log2 units
//                (two fp32 arrays, rows padded per head to a multiple of 128 with
//                LSE = +inf, D = 0); zero the fp32 dQ accumulator (and, in the
//                deterministic mode, the ordering counters).
//   main         one CTA per (b, K/V head g, 128-key tile j).  It keeps K_j, V_j in
//                shared memory and dK, dV accumulators in tensor memory for the
//                whole run, and walks every (query head of the group, 128-row
//                query tile i) pair that can see the tile (causal: query row q sits
//                at position q + Nk - Nq, so i starts where a row reaches key 128 j).  Per
//                pair, five tcgen05 GEMMs (M = 128):
//                  S^T  = K_j Q_i^T        (TMEM, fp32)
//                  dP^T = V_j dO_i^T       (TMEM, fp32)
//                  P^T  = exp2(S^T * scale*log2e - lse2_i)     (bf16, over S^T in TMEM)
//                  dS^T = P^T * (dP^T - D_i) * scale           (bf16, in shared memory)
//                  dV  += P^T dO_i  (A from TMEM),  dK += dS^T Q_i  (A from shared memory)
//                  dQ_i = dS K_j  (d = 128: as dQ_i^T = K_j^T dS^T, so that a TMEM lane
//                                  is a head-dim column; TMEM, then fp32 reductions
//                                  into the dQ accumulator)
//                Grouped heads (GQA) share K_j/V_j, so dK/dV are summed over the
//                group inside the CTA, in a fixed order, without atomics.
//   postprocess  dQ accumulator (already scaled) -> bf16.
//
// The dQ accumulation over key tiles is the only cross-CTA sum.  Default: fp32
// reductions (coalesced red.global.add.f32 for d = 128, red.global.add.v4.f32 for
// d = 64) in whatever order CTAs reach them.
// Deterministic mode (FA4's deterministic backward, wiki 未解決の問い): the CTA
// of key tile j waits (bounded) until the key tiles ranked before it have added
// their part of query tile i, then adds its part with the same reductions, fences
// them and releases the next tile: one contributor at a time in a fixed order, so
// results are bit-identical from run to run.  The order, the CTA schedule and each
// CTA's walk over its query tiles are chosen so that a CTA's predecessor was
// scheduled no later and reaches the query tile no later (see the work-unit mapping).
//
// Warp roles of the main kernel (512 threads, 16 warps):
//   warps 0-3   compute, query columns 0-63 of each tile (thread = key row = TMEM lane)
//   warps 4-7   compute, query columns 64-127
//   warps 8-11  dQ read-out and reduction; at the end the dK/dV epilogue
//   warp 12     MMA issuer (the warp runs the loop converged, lane 0 issues) and
//               TMEM allocator
//   warp 13     TMA producer (one thread)
//   warps 14-15 idle
// Tensor memory (512 columns): dV | dK | S^T (later P^T) | dP^T (then dQ_i).
#include <algorithm>
#include <type_traits>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

template <int D>
struct BwdCfg {
  static constexpr int TILE = 128 * D * 2;  // one 128 x D bf16 tile
  static constexpr int CHUNKS = D / 64;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;      // two stages
  static constexpr int OFF_DO = 4 * TILE;     // two stages
  static constexpr int OFF_DS = 6 * TILE;     // dS^T, 128 keys x 128 queries bf16, M-major, 128B swizzle
  static constexpr int OFF_LD = OFF_DS + 32768;  // two stages of lse2[128] then D[128] (fp32)
  static constexpr int OFF_BAR = OFF_LD + 2048;
  static constexpr int NBAR = 12;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static constexpr uint32_t COL_DV = 0, COL_DK = D, COL_S = 2 * D, COL_DP = 2 * D + 128;
  // d = 128: dQ is produced transposed (TMEM lane = head-dim column) for coalesced reductions
  static constexpr bool DQ_T = (D == 128);
};

// DET: compiled for the deterministic mode (launched when p.deterministic is set).  The two
// instances differ only in the dQ read-out at d = 128 (see there); elsewhere the mode is the
// run-time flag.
template <int D, bool DET>
__global__ void __launch_bounds__(512, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(p.status, 0, -5);
    return;
  }
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t kv_full = bar0;
  auto st_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto st_empty = [&](int s) { return bar0 + 8u * (3 + s); };
  const uint32_t s_full = bar0 + 8u * 5, dp_full = bar0 + 8u * 6, p_ready = bar0 + 8u * 7;
  const uint32_t ds_ready = bar0 + 8u * 8, dq_full = bar0 + 8u * 9, dq_empty = bar0 + 8u * 10;
  const uint32_t mma_done = bar0 + 8u * 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const Abort ab{abort, p.status, p.kabort, p.gen};

  // ---- work unit
  const int N = p.Nq;  // query rows; keys: p.Nk
  // Query rows are padded per head to Np, a multiple of 128, in the workspace arrays (lse2, D,
  // dQ accumulator); the last tiles of Q, dO (past Nq) and K, V (past Nk) read zeros (TMA
  // out-of-bounds fill).
  const int Np = (N + 127) & ~127;
  const int nq = Np / 128;
  const int BG = p.B * p.Hkv;
  // CTA order: groups of (up to) 8 K/V heads, key tiles heaviest first (j = 0) within a
  // group.  The CTAs resident at any time then share few heads' Q/dO tiles and dQ
  // accumulator lines, which stay in L2 (about 14% faster than key-tile-major order
  // over all heads on the B4 H16 N8192 workload).
  constexpr int kHeadGroup = 8;
  const int nkv = (p.Nk + 127) / 128;
  const int gi = blockIdx.x / (kHeadGroup * nkv);
  const int gsz = min(kHeadGroup, BG - gi * kHeadGroup);
  const int rem = blockIdx.x - gi * kHeadGroup * nkv;
  const int grp = p.H / p.Hkv;
  // Deterministic causal mode, two schedules (default mode: heaviest key tiles first, query
  // tiles ascending head by head, contributions in any order):
  //  * one query head per K/V head: contributions in descending key-tile order, lightest key
  //    tiles scheduled first, query tiles ascending.  Key tile j+1, which j waits for, started
  //    earlier and reaches every query tile one step before j, so each hand-over overlaps a
  //    step of work; the heaviest CTAs run last.
  //  * grouped heads: contributions in ascending key-tile order, heaviest first, query tiles
  //    descending from the last with the group's heads interleaved, so (h, i) is step
  //    grp (nq - 1 - i) + h of every key tile's walk and key tile j-1 (scheduled no later)
  //    reaches it at the same step as j: the hand-overs of one query tile follow each other
  //    (a skew of up to one hand-over per key tile), but the long CTAs of a group start first.
  // Measured (deterministic over default backward): causal B4 H16 N8192 +9% with the first,
  // +28% with the second; GQA B2 Hq32 Hkv8 N16384 +41% with the first, +11% with the second.
  const bool det_causal = p.deterministic && p.causal;
  const bool desc = det_causal && grp == 1;
  const bool interleave = det_causal && grp > 1;
  const int j = desc ? nkv - 1 - rem / gsz : rem / gsz;
  const int bg = gi * kHeadGroup + rem % gsz;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  // causal: query row q sits at position q + qoff; the first query tile with a row at or after
  // key 128 j is the first i with 128 i + 127 + qoff >= 128 j
  const int first = 128 * j - 127 - p.qoff;
  const int i0 = (p.causal && first > 0) ? (first + 127) / 128 : 0;
  const int ni = max(nq - i0, 0);
  const int ntiles = grp * ni;
  auto tile_head = [&](int t) { return b * p.H + g * grp + (interleave ? t % grp : t / ni); };  // b*H + h
  auto tile_row = [&](int t) { return interleave ? nq - 1 - t / grp : i0 + t % ni; };         // query tile i

  if (warp == 0 && lane == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(st_full(s), 1);
      mbar_init(st_empty(s), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(mma_done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 13 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 13) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
      for (int ch = 0; ch < C::CHUNKS; ++ch) {
        tma_load_3d(sbase + C::OFF_K + ch * 16384, &tm_k, kv_full, ch * 64, j * 128, bg);
        tma_load_3d(sbase + C::OFF_V + ch * 16384, &tm_v, kv_full, ch * 64, j * 128, bg);
      }
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t & 1;
        if (p.debug_hook == 2 && t == 1) continue;  // failure-injection test hook (never set in normal use)
        if (!mbar_wait(st_empty(s), ((t >> 1) & 1) ^ 1, ab)) break;
        const int bh = tile_head(t), i = tile_row(t);
        mbar_arrive_expect_tx(st_full(s), 2 * C::TILE + 1024);
        for (int ch = 0; ch < C::CHUNKS; ++ch) {
          tma_load_3d(sbase + C::OFF_Q + s * C::TILE + ch * 16384, &tm_q, st_full(s), ch * 64, i * 128, bh);
          tma_load_3d(sbase + C::OFF_DO + s * C::TILE + ch * 16384, &tm_do, st_full(s), ch * 64, i * 128, bh);
        }
        const size_t row0 = (size_t)bh * Np + (size_t)i * 128;
        bulk_load(sbase + C::OFF_LD + s * 1024, p.lse2 + row0, 512, st_full(s));
        bulk_load(sbase + C::OFF_LD + s * 1024 + 512, p.dvec + row0, 512, st_full(s));
        issued = t + 1;
      }
      if (*abort) {  // let copies in flight land before the CTA exits (bounded)
        for (int t = max(0, issued - 2); t < issued; ++t) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(st_full(t & 1), (t >> 1) & 1) && globaltimer() - t0 < 1000000ull) {
          }
        }
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(kv_full, 0) && globaltimer() - t0 < 1000000ull) {
        }
      }
    }
  } else if (warp == 12) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged; lane 0 issues the MMAs and commits.
    const uint32_t leader = (lane == 0) ? 1u : 0u;
    constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idKV = idesc_bf16_f32(128, D, false, true);
    constexpr uint32_t idQ = idesc_bf16_f32(128, D, true, true);
    constexpr uint32_t idQT = idesc_bf16_f32(128, 128, true, true);
    auto ss_kmajor = [&](uint32_t dcol, uint32_t a, uint32_t bsm) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_ss(tmem + dcol, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(bsm + off, 16, 1024), idS, kk > 0, leader);
      }
    };
    // D[128 keys x D] += A^T(TMEM, P^T or dS^T) * B(smem, M... [queries][D], MN-major)
    auto ts_acc = [&](uint32_t dcol, uint32_t acol, uint32_t bsm, bool acc) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tmem + dcol, tmem + acol + 64 * (kk >> 2) + (kk & 3) * 8, sdesc_sw128(bsm + kk * 2048, 16384, 1024),
               idKV, (acc || kk > 0) ? 1u : 0u, leader);
    };
    const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sDS = sbase + C::OFF_DS;
    auto sQ = [&](int s) { return sbase + C::OFF_Q + s * C::TILE; };
    auto sDO = [&](int s) { return sbase + C::OFF_DO + s * C::TILE; };
    bool ok = ntiles > 0;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(kv_full, 0, ab));
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(st_full(0), 0, ab));
    if (ok) {
      tc_fence_after();
      ss_kmajor(C::COL_S, sK, sQ(0));
      mma_commit(s_full, leader);
      ss_kmajor(C::COL_DP, sV, sDO(0));
      mma_commit(dp_full, leader);
    }
    // one query tile; MORE: another tile follows (the last iteration is peeled so that the
    // test is not a run-time branch of the issue loop)
    auto step = [&](int t, auto more_tiles) -> bool {
      constexpr bool MORE = decltype(more_tiles)::value;
      const int s = t & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(p_ready, t & 1, ab))) return false;
      tc_fence_after();
      ts_acc(C::COL_DV, C::COL_S, sDO(s), t > 0);  // dV += P^T dO_t
      if constexpr (MORE) {
        if (!__all_sync(0xffffffffu, mbar_wait(st_full(s ^ 1), ((t + 1) >> 1) & 1, ab))) return false;
        tc_fence_after();
        ss_kmajor(C::COL_S, sK, sQ(s ^ 1));  // S^T of the next tile (P^T_t already consumed)
        mma_commit(s_full, leader);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(ds_ready, t & 1, ab))) return false;
      tc_fence_after();
      // dQ first, so its read-out overlaps the dK MMA
      if constexpr (C::DQ_T) {
        // dQ_t^T = K_j^T dS^T (M = d, N = queries) into the dP^T columns: TMEM lane = head-dim
        // column, so the read-out warps reduce 128 contiguous bytes per instruction
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + C::COL_DP, sdesc_sw128(sK + kk * 2048, 16384, 1024),
                 sdesc_sw128(sDS + kk * 2048, 16384, 1024), idQT, kk > 0, leader);
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // dQ_t = dS K_j, into the dP^T columns
          mma_ss(tmem + C::COL_DP, sdesc_sw128(sDS + kk * 2048, 16384, 1024),
                 sdesc_sw128(sK + kk * 2048, 16384, 1024), idQ, kk > 0, leader);
      }
      mma_commit(dq_full, leader);
      // dK += dS^T Q_t, with dS^T read from shared memory as a K-major operand (rows = keys,
      // 64 queries per 128-byte swizzled row chunk): the same bytes the dQ MMA reads
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem + C::COL_DK, sdesc_sw128(sDS + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
               sdesc_sw128(sQ(s) + kk * 2048, 16384, 1024), idKV, (t > 0 || kk > 0) ? 1u : 0u, leader);
      mma_commit(st_empty(s), leader);
      if constexpr (MORE) {
        if (!__all_sync(0xffffffffu, mbar_wait(dq_empty, t & 1, ab))) return false;
        tc_fence_after();
        ss_kmajor(C::COL_DP, sV, sDO(s ^ 1));
        mma_commit(dp_full, leader);
      }
      return true;
    };
    for (int t = 0; ok && t + 1 < ntiles; ++t) ok = step(t, std::true_type{});
    if (ok && ntiles > 0) ok = step(ntiles - 1, std::false_type{});
    // drain: every MMA issued above has finished before TMEM is released (bounded, and
    // waited for even after an abort)
    mma_commit(mma_done, leader);
    {
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(mma_done, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
    __syncwarp();
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
    const bool key_pad = j * 128 + r >= p.Nk;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t & 1;
      // causal: key 128 j + r is masked for query 128 i + 64 w + c when it lies after the
      // query's position, i.e. for c < cut (cut <= 0: nothing masked in this half row)
      const int cut = p.causal ? r + 128 * (j - tile_row(t)) - 64 * w - p.qoff : 0;
      // this half's 64 queries: lse2 and D, four per 16-byte shared load
      const float4* lse4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 1024) + 16 * w;
      const float4* d4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 1024 + 512) + 16 * w;
      if (!__all_sync(0xffffffffu, mbar_wait(s_full, t & 1, ab))) break;
      tc_fence_after();
      float pv[64];
      {
        uint32_t ra[32], rb[32];
        tmem_ld32_nowait(tS, ra);
        tmem_wait_ld(ra);
        tmem_ld32_nowait(tS + 32, rb);  // in flight while the first 32 columns are processed
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
      if (key_pad) {  // a key row past Nk (zero-filled K) carries no probability
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
      mbar_arrive(p_ready);

      if (!__all_sync(0xffffffffu, mbar_wait(dp_full, t & 1, ab))) break;
      tc_fence_after();
      {
        uint32_t ra[32], rb[32];
        tmem_ld32_nowait(tDP, ra);
        tmem_wait_ld(ra);
        tmem_ld32_nowait(tDP + 32, rb);  // in flight while the first 32 columns are processed
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          if (cc == 1) tmem_wait_ld(rb);
          const uint32_t* src = cc ? rb : ra;
          uint32_t pk[16];
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 Dv = d4[8 * cc + c4];
            const int o = 4 * c4, q = 32 * cc + 4 * c4;
            // dS = P * (dP - D) * scale, two columns per packed op
            const uint64_t a = f2_add(f2_pack(__uint_as_float(src[o]), __uint_as_float(src[o + 1])), f2_pack(-Dv.x, -Dv.y));
            const uint64_t b = f2_add(f2_pack(__uint_as_float(src[o + 2]), __uint_as_float(src[o + 3])),
                                      f2_pack(-Dv.z, -Dv.w));
            const float2 d01 = f2_unpack(f2_mul(f2_mul(a, f2_pack(pv[q], pv[q + 1])), scx2));
            const float2 d23 = f2_unpack(f2_mul(f2_mul(b, f2_pack(pv[q + 2], pv[q + 3])), scx2));
            pk[2 * c4] = pack_bf16x2(d01.x, d01.y);
            pk[2 * c4 + 1] = pack_bf16x2(d23.x, d23.y);
          }
          // dS^T row r, queries [32cc, 32cc+32) of this half: four 16-byte pieces, 128B-swizzled
#pragma unroll
          for (int pc = 0; pc < 4; ++pc) {
            const int piece = 4 * cc + pc;
            *reinterpret_cast<uint4*>(ds_row + ((piece ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * pc], pk[4 * pc + 1], pk[4 * pc + 2], pk[4 * pc + 3]);
          }
        }
      }
      fence_async_smem();  // dS^T visible to the MMAs (async proxy)
      tc_fence_before();   // our TMEM loads of dP^T are done before the dQ MMA overwrites it
      mbar_arrive(ds_ready);
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ read-out, dK/dV epilogue
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDQ = tmem + lane_off + C::COL_DP;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int bh = tile_head(t), i = tile_row(t);
      ok = __all_sync(0xffffffffu, mbar_wait(dq_full, t & 1, ab));
      if (!ok) break;
      tc_fence_after();
      int* counter = p.deterministic ? p.counters + ((size_t)bh * nq + i) : nullptr;
      // this key tile's place in the fixed order of query tile i's contributions: ascending
      // j, or descending from the last key tile that query tile i sees (see the schedules)
      const int rank = desc ? min(nkv - 1, (128 * i + 127 + p.qoff) / 128) - j : j;
      if (p.deterministic && !(C::DQ_T && !DET)) {
        // wait for the contributions ranked before this one (the d = 128 read-out of the
        // other instance waits inside its own block)
        if (r == 0) {
          const uint64_t t0 = globaltimer();
          while (ld_acquire(counter) != rank) {
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
      if constexpr (C::DQ_T) {
        // thread r holds column r of dQ_i (rows q = 0..127).
        float* col = p.dq_acc + ((size_t)bh * Np + (size_t)i * 128) * D + r;
        if constexpr (!DET) {
          // All 128 values are read first and the TMEM columns handed back to the MMA warp at
          // once (its next dP^T MMA waits for them), then reduced: the whole backward of causal
          // B4 H16 N8192 2.87 -> 2.71 ms, GQA B2 Hq32 N16384 10.79 -> 10.06 ms.  A few values pass
          // through local memory (the kernel has 128 registers per thread); forms of this block
          // that spilled elsewhere in the kernel instead measured slower, so it is kept as it
          // is, deterministic wait included (never taken in this instance, which runs only
          // with p.deterministic == 0).
          uint32_t v0[32], v1[32], v2[32], v3[32];
          tmem_ld32_nowait(tDQ, v0);
          tmem_ld32_nowait(tDQ + 32, v1);
          tmem_ld32_nowait(tDQ + 64, v2);
          tmem_ld32_nowait(tDQ + 96, v3);
          tmem_wait_ld(v0);
          tmem_wait_ld(v1);
          tmem_wait_ld(v2);
          tmem_wait_ld(v3);
          tc_fence_before();
          mbar_arrive(dq_empty);
          if (p.deterministic) {  // wait for the contributions ranked before this one
            if (r == 0) {
              const uint64_t t0 = globaltimer();
              while (ld_acquire(counter) != rank) {
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
          if (!p.deterministic || !*abort) {
#pragma unroll
            for (int m = 0; m < 32; ++m) red_add(col + (size_t)m * D, __uint_as_float(v0[m]));
#pragma unroll
            for (int m = 0; m < 32; ++m) red_add(col + (size_t)(32 + m) * D, __uint_as_float(v1[m]));
#pragma unroll
            for (int m = 0; m < 32; ++m) red_add(col + (size_t)(64 + m) * D, __uint_as_float(v2[m]));
#pragma unroll
            for (int m = 0; m < 32; ++m) red_add(col + (size_t)(96 + m) * D, __uint_as_float(v3[m]));
          }
        } else
        // deterministic instance: read rows 0-63, reduce them, read rows 64-127, hand the TMEM
        // columns back, reduce (the order above measured 25% slower in this mode: 3.89 vs
        // 3.11 ms on causal B4 H16 N8192)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t va[32], vb[32];
          tmem_ld32_nowait(tDQ + 64 * half, va);
          tmem_ld32_nowait(tDQ + 64 * half + 32, vb);
          tmem_wait_ld(va);
          tmem_wait_ld(vb);
          if (half == 1) {
            tc_fence_before();
            mbar_arrive(dq_empty);
          }
          float* c0 = col + (size_t)(64 * half) * D;
          // deterministic mode: this CTA is the only one adding to query tile i right now (the
          // counter orders the contributions), so the reductions land in a fixed order too;
          // after a timeout nothing is added
          if (!p.deterministic || !*abort) {
#pragma unroll
            for (int m = 0; m < 32; ++m) red_add(c0 + (size_t)m * D, __uint_as_float(va[m]));
#pragma unroll
            for (int m = 0; m < 32; ++m) red_add(c0 + (size_t)(32 + m) * D, __uint_as_float(vb[m]));
          }
        }
      } else {
        float* dst = p.dq_acc + ((size_t)bh * Np + (size_t)i * 128 + r) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tDQ + 32 * c, v);
          if (c == D / 32 - 1) {
            tc_fence_before();
            mbar_arrive(dq_empty);
          }
          if (!p.deterministic || !*abort) {  // ordered in deterministic mode, as above
#pragma unroll
            for (int m = 0; m < 8; ++m)
              red_add_v4(dst + 32 * c + 4 * m, __uint_as_float(v[4 * m]), __uint_as_float(v[4 * m + 1]),
                         __uint_as_float(v[4 * m + 2]), __uint_as_float(v[4 * m + 3]));
          }
        }
      }
      if (p.deterministic) {
        __threadfence();
        named_bar(1, 128);
        // (failure-injection test hook: the first CTA keeps its successors waiting)
        if (r == 0 && !(p.debug_hook == 1 && blockIdx.x == 0)) st_release(counter, rank + 1);
      }
    }
    // mma_done is committed after every MMA of the CTA, the last dK one included
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(mma_done, 0, ab));
    if (ok) {
      tc_fence_after();
      const size_t krow = (size_t)bg * p.Nk + (size_t)j * 128 + r;
      const bool krow_valid = j * 128 + r < p.Nk;  // the last key tile may run past Nk
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

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- preprocess
// Per (padded) query row: D = sum_c dO_c * O_c (fp32 products of bf16 inputs) and
// lse2 = LSE * log2(e); rows past N of each head get lse2 = +inf (so P = 0 there) and D = 0.
// A warp takes four rows at a time, eight lanes per row, 16-byte loads.  Then zero the dQ
// accumulator (padded rows included) and the counters.
FA_DEV float dot_bf16x8(uint4 x, uint4 y, float acc) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    acc = fmaf(__uint_as_float(xs[k] << 16), __uint_as_float(ys[k] << 16), acc);
    acc = fmaf(__uint_as_float(xs[k] & 0xffff0000u), __uint_as_float(ys[k] & 0xffff0000u), acc);
  }
  return acc;
}

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                                      const float* __restrict__ lse, float* __restrict__ lse2,
                                                      float* __restrict__ dvec,
                                                      float4* __restrict__ dq_acc, int* __restrict__ counters,
                                                      long long heads, int N, int Np, long long n_counters) {
  constexpr int V = D / 64;  // 16-byte vectors per lane (eight lanes per row)
  const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
  const long long gw = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const long long quads = heads * Np / 4;  // Np is a multiple of 128, so a quad stays in one head
  for (long long qd = gw; qd < quads; qd += nwarps) {
    const long long prow = 4 * qd + (lane >> 3);
    long long row = prow;
    bool valid = true;
    if (N != Np) {
      const long long bh = prow / Np;
      const int n = static_cast<int>(prow - bh * Np);
      valid = n < N;
      row = bh * N + n;
    }
    float acc = 0.f;
    if (valid) {
      const uint4* a = reinterpret_cast<const uint4*>(o + row * D) + sub * V;
      const uint4* c = reinterpret_cast<const uint4*>(dout + row * D) + sub * V;
      uint4 xa[V], xc[V];
#pragma unroll
      for (int k = 0; k < V; ++k) {
        xa[k] = a[k];
        xc[k] = c[k];
      }
#pragma unroll
      for (int k = 0; k < V; ++k) acc = dot_bf16x8(xa[k], xc[k], acc);
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0) {
      lse2[prow] = valid ? lse[row] * 1.4426950408889634f : INFINITY;
      dvec[prow] = valid ? acc : 0.f;
    }
  }
  const long long n4 = heads * Np * D / 4;
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthr = (long long)gridDim.x * blockDim.x;
  for (long long k = tid; k < n4; k += nthr) dq_acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (counters)
    for (long long k = tid; k < n_counters; k += nthr) counters[k] = 0;
}

// ---------------------------------------------------------------- postprocess
// dQ (bf16, [heads][N][d]) = accumulator (fp32, [heads][Np][d]; the softmax scale is already
// folded into dS).
__global__ void __launch_bounds__(256) bwd_post_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq, long long n4,
                                                       int d4, int N, int Np) {
  const long long nthr = (long long)gridDim.x * blockDim.x;
  for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < n4; k += nthr) {
    long long src = k;
    if (N != Np) {
      const long long row = k / d4;
      const long long bh = row / N;
      src = ((bh * Np + (row - bh * N)) * d4) + (k - row * d4);
    }
    const float4 x = acc[src];
    dq[k] = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
  }
}

static int sm_count() {
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

cudaError_t launch_bwd_pre(int d, const void* o, const void* dout, const float* lse, float* lse2, float* dvec,
                           float* dq_acc, int* counters, long long heads, int N, long long n_counters,
                           cudaStream_t stream) {
  const int Np = (N + 127) & ~127;
  const long long want = (heads * Np / 4 + 7) / 8;
  const int grid = (int)std::min<long long>(std::max<long long>(want, 1), (long long)sm_count() * 8);
  if (d == 64)
    bwd_pre_kernel<64><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                                                 lse, lse2, dvec, reinterpret_cast<float4*>(dq_acc), counters, heads,
                                                 N, Np, n_counters);
  else if (d == 128)
    bwd_pre_kernel<128><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                                                  lse, lse2, dvec, reinterpret_cast<float4*>(dq_acc), counters, heads,
                                                  N, Np, n_counters);
  else
    bwd_pre_kernel<256><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                                                  lse, lse2, dvec, reinterpret_cast<float4*>(dq_acc), counters, heads,
                                                  N, Np, n_counters);
  return cudaGetLastError();
}

cudaError_t launch_bwd_post(const float* dq_acc, void* dq, long long heads, int N, int d, cudaStream_t stream) {
  const int Np = (N + 127) & ~127;
  const long long n4 = heads * N * d / 4;
  const int grid = (int)std::min<long long>(std::max<long long>((n4 + 255) / 256, 1), (long long)sm_count() * 8);
  bwd_post_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(dq_acc), static_cast<uint2*>(dq), n4,
                                            d / 4, N, Np);
  return cudaGetLastError();
}

template <int D, bool DET>
static cudaError_t launch_bwd_main_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(bwd_main_kernel<D, DET>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const long long blocks = (long long)((p.Nk + 127) / 128) * p.B * p.Hkv;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  bwd_main_kernel<D, DET><<<dim3((unsigned)blocks), dim3(512), C::SMEM, stream>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
  if (d == 64)
    return p.deterministic ? launch_bwd_main_d<64, true>(tq, tk, tv, tdo, p, stream)
                           : launch_bwd_main_d<64, false>(tq, tk, tv, tdo, p, stream);
  return p.deterministic ? launch_bwd_main_d<128, true>(tq, tk, tv, tdo, p, stream)
                         : launch_bwd_main_d<128, false>(tq, tk, tv, tdo, p, stream);
}

}  // namespace fa
