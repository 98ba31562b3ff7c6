// fa_bwd256.cu -- the attention backward's main stage at head dimension 256.
//
// The method is fa_bwd.cu's (P recomputed from the saved LSE: the explainer's recomputation
// paragraph; the gradient of L = sum(O * dO)).  At d = 256 the dK and dV accumulators of a
// 128-key tile would fill all 512 tensor-memory columns, so the head dimension is split: a
// pair of CTAs per (b, K/V head, 128-key tile), CTA h owning head-dimension columns
// [128 h, 128 h + 128).  Both recompute S^T = K Q^T and dP^T = V dO^T over all 256 columns
// (that work is done twice); each accumulates its half of dV, dK and adds its half of dQ.
// Per (query head of the group, 64-row query tile i):
//
//   S^T  = K_j Q_i^T                (M = 128 keys, N = 64, K = 256)      TMEM
//   dP^T = V_j dO_i^T               (M = 128, N = 64, K = 256; A = V_j from TMEM)
//   P^T  = exp2(S^T scale log2e - lse2_i)  (bf16, over S^T)
//   dS^T = P^T (dP^T - D_i) scale          (bf16, shared memory)
//   dV_h += P^T dO_i[:, h]          (M = 128, N = 128, K = 64; A from TMEM)
//   dK_h += dS^T Q_i[:, h]          (M = 128, N = 128, K = 64)
//   dQ_i[:, h]^T = K_j[:, h]^T dS^T (M = 128, N = 64, K = 128 keys), into the dP^T columns,
//                  read out and added with coalesced fp32 reductions (in a fixed order in
//                  deterministic mode, one ordering counter per (head, query tile, half))
//
// V_j is read by one GEMM only, so it lives in tensor memory (written once per CTA by the
// compute warps from plain loads) as dP^T's A operand.  That leaves K_j and two stages of
// Q_i and dO_i (32 KB each per stage) in shared memory, so the next tile's copies overlap the
// current tile.  The MMA warp issues, per tile t:
//   dV(t) | S^T(t+1) | dQ^T(t), dK(t) | dP^T(t+1) once dQ^T(t) has been read out
// so the compute warps' P pass of tile t+1 overlaps the dQ and dK MMAs of tile t.
//
// Warp roles (512 threads): warps 0-7 compute (warpgroup w: queries 32 w .. 32 w + 31 of the
// tile, thread = key row = TMEM lane), warps 8-11 dQ read-out then the dK/dV epilogue, warp 12
// MMA issue and TMEM allocation, warp 13 TMA producer, warps 14-15 idle.
// Tensor memory: dV_h | dK_h | S^T (then P^T) | dP^T (then dQ^T_h) | V_j (512 columns).
#include <algorithm>
#include <type_traits>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

struct Bwd256Cfg {
  static constexpr int D = 256;
  static constexpr int OFF_K = 0;        // K_j [128 keys][256 d]: four chunks [128][64] of 16 KB
  static constexpr int OFF_Q = 65536;    // two stages of Q_i [64 rows][256 d]: four chunks [64][64] of 8 KB
  static constexpr int OFF_DO = 131072;  // two stages of dO_i, same layout
  static constexpr int STAGE = 32768;
  static constexpr int OFF_DS = 196608;  // dS^T [128 keys][64 queries]: one 16 KB chunk
  static constexpr int OFF_LD = 212992;  // two stages of lse2[64] then D[64] (fp32)
  static constexpr int OFF_BAR = 214016;
  static constexpr int NBAR = 14;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static constexpr uint32_t COL_DV = 0, COL_DK = 128, COL_S = 256, COL_DP = 320, COL_V = 384;
};

__global__ void __launch_bounds__(512, 1)
    bwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using C = Bwd256Cfg;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, -5);
    return;
  }
  const uint32_t bar0 = sbase + C::OFF_BAR;
  const uint32_t k_full = bar0;
  auto st_full = [&](int s) { return bar0 + 8u + 8u * s; };    // Q, dO, lse2/D of one stage
  auto st_empty = [&](int s) { return bar0 + 24u + 8u * s; };
  const uint32_t s_full = bar0 + 40, dp_full = bar0 + 48, p_ready = bar0 + 56, ds_ready = bar0 + 64;
  const uint32_t dq_full = bar0 + 72, dq_empty = bar0 + 80, v_ready = bar0 + 88, mma_done = bar0 + 96;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const Abort ab{abort, p.status, p.kabort, p.gen};

  // ---- work unit: (b, K/V head g, key tile j, head-dimension half h); both halves of a key
  // tile are adjacent CTAs, groups of 8 K/V heads, key tiles heaviest first (as fa_bwd.cu)
  const int N = p.Nq;
  const int Np = (N + 127) & ~127;
  const int nq = Np / 64;  // 64-row query tiles
  const int BG = p.B * p.Hkv;
  constexpr int kHeadGroup = 8;
  const int nkv = (p.Nk + 127) / 128;
  const int hh = blockIdx.x & 1;
  const int cta = blockIdx.x >> 1;
  const int gi = cta / (kHeadGroup * nkv);
  const int gsz = min(kHeadGroup, BG - gi * kHeadGroup);
  const int rem = cta - gi * kHeadGroup * nkv;
  const int grp = p.H / p.Hkv;
  // deterministic causal schedules as in fa_bwd.cu
  const bool det_causal = p.deterministic && p.causal;
  const bool desc = det_causal && grp == 1;
  const bool interleave = det_causal && grp > 1;
  const int j = desc ? nkv - 1 - rem / gsz : rem / gsz;
  const int bg = gi * kHeadGroup + rem % gsz;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  // causal: the first 64-row query tile with a row at or after key 128 j
  const int first = 128 * j - 63 - p.qoff;
  const int i0 = (p.causal && first > 0) ? (first + 63) / 64 : 0;
  const int ni = max(nq - i0, 0);
  const int ntiles = grp * ni;
  auto tile_head = [&](int t) { return b * p.H + g * grp + (interleave ? t % grp : t / ni); };
  auto tile_row = [&](int t) { return interleave ? nq - 1 - t / grp : i0 + t % ni; };

  if (warp == 0 && lane == 0) {
    mbar_init(k_full, 1);
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
    mbar_init(v_ready, 256);
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
    prefetch_tmap(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 13) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      mbar_arrive_expect_tx(k_full, 65536);
      for (int ch = 0; ch < 4; ++ch)
        tma_load_3d(sbase + C::OFF_K + ch * 16384, &tm_k, k_full, ch * 64, j * 128, bg);
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t & 1;
        if (p.debug_hook == 2 && t == 1) break;  // failure-injection test hook (never set in normal use)
        // the stage's previous tile (t - 2) is done: its dK MMA, the last reader, completed
        if (!mbar_wait(st_empty(s), ((t >> 1) & 1) ^ 1, ab)) break;
        const int bh = tile_head(t), i = tile_row(t);
        mbar_arrive_expect_tx(st_full(s), 2 * C::STAGE + 512);
        for (int ch = 0; ch < 4; ++ch) {
          tma_load_3d(sbase + C::OFF_Q + s * C::STAGE + ch * 8192, &tm_q, st_full(s), ch * 64, i * 64, bh);
          tma_load_3d(sbase + C::OFF_DO + s * C::STAGE + ch * 8192, &tm_do, st_full(s), ch * 64, i * 64, bh);
        }
        const size_t row0 = (size_t)bh * Np + (size_t)i * 64;
        bulk_load(sbase + C::OFF_LD + s * 512, p.lse2 + row0, 256, st_full(s));
        bulk_load(sbase + C::OFF_LD + s * 512 + 256, p.dvec + row0, 256, st_full(s));
        issued = t + 1;
      }
      if (*abort) {  // let copies in flight land before the CTA exits (bounded)
        for (int t = max(0, issued - 2); t < issued; ++t) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(st_full(t & 1), (t >> 1) & 1) && globaltimer() - t0 < 1000000ull) {
          }
        }
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(k_full, 0) && globaltimer() - t0 < 1000000ull) {
        }
      }
    }
  } else if (warp == 12) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 64, false, false);   // S^T, dP^T (K-major)
      constexpr uint32_t idKV = idesc_bf16_f32(128, 128, false, true);  // dV, dK (B: MN-major)
      constexpr uint32_t idQ = idesc_bf16_f32(128, 64, true, true);     // dQ^T (A, B: MN-major)
      const uint32_t sK = sbase + C::OFF_K, sDS = sbase + C::OFF_DS;
      auto sQ = [&](int t) { return sbase + C::OFF_Q + (t & 1) * C::STAGE; };
      auto sDO = [&](int t) { return sbase + C::OFF_DO + (t & 1) * C::STAGE; };
      auto issue_s = [&](int t) {  // S^T = K Q_t^T over the four head-dimension chunks
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::COL_S, sdesc_sw128(sK + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(sQ(t) + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), idS, kk > 0);
      };
      auto issue_dp = [&](int t) {  // dP^T = V dO_t^T: A = V from TMEM (16 d = 8 columns per step)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts(tmem + C::COL_DP, tmem + C::COL_V + kk * 8,
                 sdesc_sw128(sDO(t) + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), idS, kk > 0);
      };
      bool ok = mbar_wait(k_full, 0, ab) && mbar_wait(st_full(0), 0, ab);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        mma_commit(s_full);
        ok = mbar_wait(v_ready, 0, ab);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(0);
        mma_commit(dp_full);
      }
      for (int t = 0; ok && t < ntiles; ++t) {
        const uint32_t par = t & 1;
        const bool more = t + 1 < ntiles;
        if (!(ok = mbar_wait(p_ready, par, ab))) break;
        tc_fence_after();
        // dV_h += P^T dO[:, h]: A = P^T from TMEM (16 queries = 8 columns per step; queries
        // 32 w .. 32 w + 31 in columns 32 w .. 32 w + 15), B = dO's chunks 2h, 2h+1 (MN-major)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(tmem + C::COL_DV, tmem + C::COL_S + 32 * (kk >> 1) + (kk & 1) * 8,
                 sdesc_sw128(sDO(t) + 2 * hh * 8192 + kk * 2048, 8192, 1024), idKV, (t > 0 || kk > 0) ? 1u : 0u);
        if (more) {  // S^T of the next tile over the P^T columns (the dV MMAs above read them first)
          if (!(ok = mbar_wait(st_full((t + 1) & 1), ((t + 1) >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_s(t + 1);
          mma_commit(s_full);
        }
        if (!(ok = mbar_wait(ds_ready, par, ab))) break;
        tc_fence_after();
        // dQ^T_h = K[:, h]^T dS^T into the dP^T columns (read by the compute warps before
        // ds_ready): A = K's chunks 2h, 2h+1 as MN-major [keys][d] (16 KB apart), B = dS^T
        // [keys][64 queries] (MN-major)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + C::COL_DP, sdesc_sw128(sK + 2 * hh * 16384 + kk * 2048, 16384, 1024),
                 sdesc_sw128(sDS + kk * 2048, 16384, 1024), idQ, kk > 0);
        mma_commit(dq_full);
        // dK_h += dS^T Q[:, h]: A = dS^T (K-major over queries), B = Q's chunks 2h, 2h+1
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem + C::COL_DK, sdesc_sw128(sDS + kk * 32, 16, 1024),
                 sdesc_sw128(sQ(t) + 2 * hh * 8192 + kk * 2048, 8192, 1024), idKV, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(st_empty(t & 1));  // Q, dO and the lse2/D rows of this stage are free after these
        if (more) {  // dP^T of the next tile, once dQ^T(t) has left the columns
          if (!(ok = mbar_wait(dq_empty, par, ab) && mbar_wait(st_full((t + 1) & 1), ((t + 1) >> 1) & 1, ab)))
            break;
          tc_fence_after();
          issue_dp(t + 1);
          mma_commit(dp_full);
        }
      }
      mma_commit(mma_done);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(mma_done, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute: V, then P^T and dS^T
    const int w = warp >> 2;           // query quarter: queries 32 w .. 32 w + 31 of the tile
    const int r = threadIdx.x & 127;   // key row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool key_pad = j * 128 + r >= p.Nk;
    if (ntiles > 0) {
      // V row r into TMEM (A operand of dP^T): warpgroup w writes head-dimension columns
      // [128 w, 128 w + 128), two bf16 per 32-bit column; rows past Nk are zero
      const uint4* vrow = static_cast<const uint4*>(p.v) + ((size_t)bg * p.Nk + (size_t)j * 128 + r) * (D / 8) + 16 * w;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint4 x = key_pad ? make_uint4(0u, 0u, 0u, 0u) : ld_nc_v4(vrow + 8 * half + m);
          pk[4 * m] = x.x;
          pk[4 * m + 1] = x.y;
          pk[4 * m + 2] = x.z;
          pk[4 * m + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + C::COL_V + 64 * w + 32 * half, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(v_ready);
    }
    const uint32_t tS = tmem + lane_off + C::COL_S + 32 * w;
    const uint32_t tDP = tmem + lane_off + C::COL_DP + 32 * w;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t scx2 = f2_pack(p.scale, p.scale);
    uint8_t* ds_row = smem + C::OFF_DS + r * 128;
    for (int t = 0; t < ntiles; ++t) {
      // causal: key 128 j + r is masked for query 64 i + 32 w + c when c < cut
      const int cut = p.causal ? r + 128 * j - 64 * tile_row(t) - 32 * w - p.qoff : 0;
      const int s = t & 1;
      // lse2/D of this stage: landed with the stage's copies, which the MMA warp waited for
      // before S^T(t)
      const float4* lse4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 512) + 8 * w;
      const float4* d4 = reinterpret_cast<const float4*>(smem + C::OFF_LD + s * 512 + 256) + 8 * w;
      if (!__all_sync(0xffffffffu, mbar_wait(s_full, t & 1, ab))) break;
      tc_fence_after();
      float pv[32];
      {
        uint32_t ra[32];
        tmem_ld32(tS, ra);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 L = lse4[c4];
          const int o = 4 * c4;
          const float2 x01 = f2_unpack(f2_fma(f2_pack(__uint_as_float(ra[o]), __uint_as_float(ra[o + 1])), sl2x2,
                                              f2_pack(-L.x, -L.y)));
          const float2 x23 = f2_unpack(f2_fma(f2_pack(__uint_as_float(ra[o + 2]), __uint_as_float(ra[o + 3])), sl2x2,
                                              f2_pack(-L.z, -L.w)));
          pv[o] = ex2_mufu(x01.x);
          pv[o + 1] = ex2_mufu(x01.y);
          pv[o + 2] = ex2_mufu(x23.x);
          pv[o + 3] = ex2_mufu(x23.y);
        }
      }
      if (key_pad) {
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[c] = 0.f;
      }
      if (cut > 0) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c < cut) pv[c] = 0.f;
      }
      {
        uint32_t pk[16];
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) pk[c2] = pack_bf16x2(pv[2 * c2], pv[2 * c2 + 1]);
        // P^T over this warpgroup's own S^T columns (all read above): queries 32 w .. 32 w + 31
        // as bf16 pairs in columns 32 w .. 32 w + 15
        tmem_st16(tS, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_ready);

      if (!__all_sync(0xffffffffu, mbar_wait(dp_full, t & 1, ab))) break;
      tc_fence_after();
      {
        uint32_t ra[32];
        tmem_ld32(tDP, ra);
        uint32_t pk[16];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 Dv = d4[c4];
          const int o = 4 * c4;
          const uint64_t a = f2_add(f2_pack(__uint_as_float(ra[o]), __uint_as_float(ra[o + 1])), f2_pack(-Dv.x, -Dv.y));
          const uint64_t bb = f2_add(f2_pack(__uint_as_float(ra[o + 2]), __uint_as_float(ra[o + 3])),
                                     f2_pack(-Dv.z, -Dv.w));
          const float2 d01 = f2_unpack(f2_mul(f2_mul(a, f2_pack(pv[o], pv[o + 1])), scx2));
          const float2 d23 = f2_unpack(f2_mul(f2_mul(bb, f2_pack(pv[o + 2], pv[o + 3])), scx2));
          pk[2 * c4] = pack_bf16x2(d01.x, d01.y);
          pk[2 * c4 + 1] = pack_bf16x2(d23.x, d23.y);
        }
        // dS^T row r, queries 32 w .. 32 w + 31: pieces 4 w .. 4 w + 3 (8 queries each), swizzled
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const int piece = 4 * w + pc;
          *reinterpret_cast<uint4*>(ds_row + ((piece ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * pc], pk[4 * pc + 1], pk[4 * pc + 2], pk[4 * pc + 3]);
        }
      }
      fence_async_smem();  // dS^T visible to the MMAs (async proxy)
      tc_fence_before();   // our TMEM loads of dP^T are done before dQ^T overwrites the columns
      mbar_arrive(ds_ready);
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ read-out, dK/dV epilogue
    // dQ^T_h: TMEM lane L = head-dimension column 128 h + L, column c = query c of the tile
    const int L = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tDQ = tmem + lane_off + C::COL_DP;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int bh = tile_head(t), i = tile_row(t);
      ok = __all_sync(0xffffffffu, mbar_wait(dq_full, t & 1, ab));
      if (!ok) break;
      tc_fence_after();
      // hand the columns back to the MMA warp first: the next dP^T waits for them
      uint32_t va[32], vb[32];
      tmem_ld32_nowait(tDQ, va);
      tmem_ld32_nowait(tDQ + 32, vb);
      tmem_wait_ld(va);
      tmem_wait_ld(vb);
      tc_fence_before();
      mbar_arrive(dq_empty);
      // deterministic: one counter per (head, 64-row query tile, half); contributions in the
      // order of the schedule (ascending key tiles, or descending from the last one the query
      // tile sees)
      int* counter = p.deterministic ? p.counters + (((size_t)bh * nq + i) * 2 + hh) : nullptr;
      const int rank = desc ? min(nkv - 1, (64 * i + 63 + p.qoff) / 128) - j : j;
      if (p.deterministic) {
        if (L == 0) {
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
        float* col = p.dq_acc + ((size_t)bh * Np + (size_t)i * 64) * D + 128 * hh + L;
#pragma unroll
        for (int m = 0; m < 32; ++m) red_add(col + (size_t)m * D, __uint_as_float(va[m]));
#pragma unroll
        for (int m = 0; m < 32; ++m) red_add(col + (size_t)(32 + m) * D, __uint_as_float(vb[m]));
      }
      if (p.deterministic) {
        __threadfence();
        named_bar(1, 128);
        if (L == 0 && !(p.debug_hook == 1 && blockIdx.x < 2)) st_release(counter, rank + 1);
      }
    }
    if (ok && ntiles > 0) ok = __all_sync(0xffffffffu, mbar_wait(mma_done, 0, ab));
    if (ok) {
      tc_fence_after();
      const size_t krow = (size_t)bg * p.Nk + (size_t)j * 128 + L;
      const bool krow_valid = j * 128 + L < p.Nk;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(which ? p.dk : p.dv) + krow * D + 128 * hh);
        const uint32_t tcol = tmem + lane_off + (which ? C::COL_DK : C::COL_DV);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tcol + 32 * c, v);
          if (ntiles == 0) {
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

  __syncwarp();  // single-lane roles rejoin their warps before the warp-wide dealloc
  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_bwd256(const CUtensorMap& tq64, const CUtensorMap& tk, const CUtensorMap& tdo64, const BwdParams& p,
                          cudaStream_t stream) {
  using C = Bwd256Cfg;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(bwd256_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const long long blocks = 2LL * ((p.Nk + 127) / 128) * p.B * p.Hkv;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  bwd256_kernel<<<dim3((unsigned)blocks), dim3(512), C::SMEM, stream>>>(tq64, tk, tdo64, p);
  return cudaGetLastError();
}

}  // namespace fa
