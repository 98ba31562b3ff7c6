// fa_fp8.cu -- FP8 (e4m3) exact-attention forward, head dimension 128.
//
// The wiki note's FA3 item 3 (and its insight on FP8 numerical stability): FP8 inputs with
// block quantisation (one scale per block of rows instead of one per tensor) and incoherent
// processing (Q and K multiplied by a random orthogonal matrix, which leaves Q K^T unchanged
// and spreads outlier features over all head-dimension columns), with higher-precision
// accumulation.  Two kernels:
//
//   fp8_quant_kernel   per block of 128 rows of one head: optional rotation of each row by
//                      H diag(r) / sqrt(d) (a fast Walsh-Hadamard transform in fp32, stages
//                      h = 1, 2, ..., 64, pairs (a, b) -> (a + b, a - b); r the caller's signs),
//                      the block's amax, scale = amax / 448, codes = e4m3(x * 448 / amax) with
//                      round-to-nearest-even and saturation.  V is written transposed
//                      ([d][keys]) so that every MMA operand of the attention kernel is K-major.
//   fwd_fp8_kernel     the persistent forward of fa_fwd.cu on the codes: S = Q8 K8^T with
//                      tcgen05 kind::f8f6f4 MMAs (K = 32 per instruction), scaled per tile by
//                      sq * sk * softmax scale inside the exponent's FMA; an exact running max
//                      (every growth rescales, so each weight is at most 1); P quantised to
//                      e4m3 as 448 f_j p with the tile's V block scale folded in
//                      (f_j = sv_j / sv_max, a log2 offset in the same FMA); O += P8 V8 from
//                      tensor memory; O normalised by the sum of the quantised weights (summed
//                      per tile in f16, where e4m3 values are exact) and rescaled by
//                      sv_max / 448; LSE from the unquantised sum.
//
// Warp roles, tensor memory (S0 | S1 | O0 | O1) and the register split are those of fa_fwd.cu;
// tiles are 128 x 128 bytes (one 128-byte swizzle span per row).
#include <algorithm>
#include <type_traits>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

// ---------------------------------------------------------------- PTX helpers (FP8)
// Two fp32 values to a packed e4m3 pair (lo in the low byte), round-to-nearest-even, saturating.
FA_DEV uint16_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// A packed e4m3 pair widened exactly to an f16 pair.
FA_DEV uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
FA_DEV uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
FA_DEV float f16x2_sum(uint32_t v) {
  float lo, hi;
  asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, u;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(v));
  return lo + hi;
}
FA_DEV void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
FA_DEV void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor, kind::f8f6f4: fp32 accumulator, e4m3 A and B (format 0), K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- quantisation
// One CTA (8 warps) per (head, block of 128 rows); warp w takes rows 16 w .. 16 w + 15, a lane
// holds head-dimension columns 4 lane .. 4 lane + 3 of a row.
template <bool ROTATE, bool TRANSPOSE>
__global__ void __launch_bounds__(256) fp8_quant_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ out,
                                                        float* __restrict__ scales, const float* __restrict__ signs,
                                                        float inv_sqrt_d, int N, int nb, int pitch) {
  __shared__ float wmax[8];
  __shared__ __align__(16) uint8_t tile[TRANSPOSE ? 128 * 128 : 16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long head = blockIdx.x / nb;
  const int blk = blockIdx.x % nb;
  const int r0 = blk * 128;
  const int rows = min(128, N - r0);
  float v[16][4];
  // column scale of the rotation: r_j * fp32(1 / sqrt(d)), r_j = +-1 (the caller's signs)
  float cs[4] = {1.f, 1.f, 1.f, 1.f};
  if (ROTATE) {
#pragma unroll
    for (int e = 0; e < 4; ++e) cs[e] = signs[4 * lane + e] > 0.f ? inv_sqrt_d : -inv_sqrt_d;
  }
  float amax = 0.f;
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    const int row = 16 * warp + rr;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    if (row < rows) {
      const uint2 raw = *reinterpret_cast<const uint2*>(x + ((size_t)head * N + r0 + row) * 128 + 4 * lane);
      a[0] = __uint_as_float(raw.x << 16);
      a[1] = __uint_as_float(raw.x & 0xffff0000u);
      a[2] = __uint_as_float(raw.y << 16);
      a[3] = __uint_as_float(raw.y & 0xffff0000u);
      if (ROTATE) {
        // stages h = 1 and 2 inside the lane's four columns
        float t0 = a[0] + a[1], t1 = a[0] - a[1], t2 = a[2] + a[3], t3 = a[2] - a[3];
        a[0] = t0 + t2;
        a[1] = t1 + t3;
        a[2] = t0 - t2;
        a[3] = t1 - t3;
        // stages h = 4 .. 64 across lanes: the lane without bit h/4 keeps a + b, the other a - b
#pragma unroll
        for (int hl = 1; hl < 32; hl <<= 1) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float other = __shfl_xor_sync(0xffffffffu, a[e], hl);
            a[e] = (lane & hl) ? other - a[e] : a[e] + other;
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = __fmul_rn(a[e], cs[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[rr][e] = a[e];
      amax = fmaxf(amax, fabsf(a[e]));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) wmax[warp] = amax;
  __syncthreads();
  amax = wmax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, wmax[w]);
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
  if (threadIdx.x == 0) scales[head * nb + blk] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
#pragma unroll
  for (int rr = 0; rr < 16; ++rr) {
    const int row = 16 * warp + rr;
    const uint32_t lo = pack_e4m3x2(__fmul_rn(v[rr][0], inv), __fmul_rn(v[rr][1], inv));
    const uint32_t hi = pack_e4m3x2(__fmul_rn(v[rr][2], inv), __fmul_rn(v[rr][3], inv));
    const uint32_t word = lo | (hi << 16);
    if (TRANSPOSE) {
      *reinterpret_cast<uint32_t*>(tile + row * 128 + 4 * lane) = word;  // rows past N hold zero codes
    } else if (row < rows) {
      *reinterpret_cast<uint32_t*>(out + ((size_t)head * N + r0 + row) * 128 + 4 * lane) = word;
    }
  }
  if (TRANSPOSE) {
    __syncthreads();
    // out[head][dcol][key], pitch bytes per head-dimension row: thread t writes 64 keys of row t/2
    const int dcol = threadIdx.x >> 1, k0 = 64 * (threadIdx.x & 1);
    uint8_t* dst = out + ((size_t)head * 128 + dcol) * pitch + r0 + k0;
    const int nk = min(64, pitch - r0 - k0);  // keys of this block inside the padded row
    for (int k = 0; k < nk; k += 4) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) word |= static_cast<uint32_t>(tile[(k0 + k + e) * 128 + dcol]) << (8 * e);
      *reinterpret_cast<uint32_t*>(dst + k) = word;
    }
  }
}

// The largest V block scale of every head.
__global__ void __launch_bounds__(256) fp8_vmax_kernel(const float* __restrict__ sv, float* __restrict__ vmax,
                                                       long long heads, int nb) {
  const long long h = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (h >= heads) return;
  float m = 0.f;
  for (int i = lane; i < nb; i += 32) m = fmaxf(m, sv[h * nb + i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) vmax[h] = m;
}

// ---------------------------------------------------------------- attention
struct Fp8Cfg {
  static constexpr int TILE = 16384;  // 128 x 128 bytes
  static constexpr int STAGES = 8;
  static constexpr int SMEM_Q = 2 * TILE;
  static constexpr int SMEM_RING = STAGES * TILE;
  static constexpr int NBAR = 2 * STAGES + 11;
  static constexpr int SMEM_BYTES = 1024 + SMEM_Q + SMEM_RING + NBAR * 8 + 16;
  static constexpr int THREADS = 384;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 384;
  static constexpr int REG_SOFTMAX = 184, REG_OTHER = 136;  // of 168 at launch (see fa_fwd.cu)
};

struct Fp8Unit {
  int bh, q0, n_kv, kv_z;
  bool two;
};

FA_DEV int fp8_unit_index(int r) {  // boustrophedon order (see fa_fwd.cu)
  const int G = gridDim.x;
  return r * G + ((r & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
}

FA_DEV Fp8Unit fp8_unit(const Fp8Params& p, int u) {
  const int ncb = (p.N + 255) / 256;
  const int BH = p.B * p.H;
  Fp8Unit w;
  const int cb = p.causal ? (ncb - 1 - u / BH) : (u / BH);
  w.bh = u % BH;
  const int b = w.bh / p.H, h = w.bh % p.H;
  w.kv_z = b * p.Hkv + h / (p.H / p.Hkv);
  w.q0 = cb * 256;
  const int n_kv_all = (p.N + 127) / 128;
  const int last_row = min(w.q0 + 255, p.N - 1);
  w.n_kv = p.causal ? min(n_kv_all, last_row / 128 + 1) : n_kv_all;
  w.two = p.N - w.q0 > 128;
  return w;
}

__global__ void __launch_bounds__(384, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, const Fp8Params p, int n_units) {
  using C = Fp8Cfg;
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
  const int N = p.N;
  const int nb = (N + 127) / 128;

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
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 9 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_vt);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_OTHER));
    if (warp == 9 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      uint32_t it = 0, issued = 0, q_loads = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int u = fp8_unit_index(r);
        if (u >= n_units) break;
        const Fp8Unit w = fp8_unit(p, u);
        if (q_loads > 0 && !mbar_wait(q_empty, (q_loads - 1) & 1, ab)) break;
        mbar_arrive_expect_tx(q_full, 2 * C::TILE);
        for (int qt = 0; qt < 2; ++qt)
          tma_load_3d(smem_u32(sQ + qt * C::TILE), &tm_q, q_full, 0, w.q0 + qt * 128, w.bh);
        ++q_loads;
        for (int jj = 0; jj < 2 * w.n_kv; ++jj, ++it) {
          const uint32_t slot = it % C::STAGES;
          if (!mbar_wait(empty_bar(slot), ((it / C::STAGES) & 1) ^ 1, ab)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(slot), C::TILE);
          if (jj & 1)  // V^T tile: head-dimension rows, this key tile's 128 columns
            tma_load_3d(smem_u32(sRing + slot * C::TILE), &tm_vt, full_bar(slot), (jj >> 1) * 128, 0, w.kv_z);
          else
            tma_load_3d(smem_u32(sRing + slot * C::TILE), &tm_k, full_bar(slot), 0, (jj >> 1) * 128, w.kv_z);
          issued = it + 1;
        }
      }
      if (*abort) {
        for (uint32_t k = issued > C::STAGES ? issued - C::STAGES : 0; k < issued; ++k) {
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
    } else if (warp == 8 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t id = idesc_e4m3_f32(128, 128);
      const uint32_t q_addr = smem_u32(sQ), ring = smem_u32(sRing);
      auto issue_s = [&](int w, uint32_t slot) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss_f8(tmem + (w ? C::COL_S1 : C::COL_S0), sdesc_sw128(q_addr + w * C::TILE + kk * 32, 16, 1024),
                    sdesc_sw128(ring + slot * C::TILE + kk * 32, 16, 1024), id, kk > 0);
      };
      // O_w += P8_w V8^T: A = the e4m3 weights in tensor memory (four per column), B = V^T (K-major)
      auto issue_pv = [&](int w, uint32_t slot, bool acc) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_f8(tmem + (w ? C::COL_O1 : C::COL_O0), tmem + (w ? C::COL_S1 : C::COL_S0) + kk * 8,
                    sdesc_sw128(ring + slot * C::TILE + kk * 32, 16, 1024), id, (acc || kk > 0) ? 1u : 0u);
      };
      auto slot_of = [](uint32_t k) { return k % C::STAGES; };
      auto par_of = [](uint32_t k) { return (k / C::STAGES) & 1u; };
      uint32_t it = 0, units = 0, units2 = 0, jg0 = 0, jg1 = 0;
      auto unit_mma = [&](const Fp8Unit& w, auto two_tiles, const uint32_t it0, const uint32_t u_idx,
                          const uint32_t u2_idx, const uint32_t g0, const uint32_t g1) -> bool {
        constexpr bool TWO = decltype(two_tiles)::value;
        const int n_kv = w.n_kv;
        if (!mbar_wait(q_full, u_idx & 1, ab)) return false;
        if (!mbar_wait(full_bar(slot_of(it0)), par_of(it0), ab)) return false;
        tc_fence_after();
        issue_s(0, slot_of(it0));
        mma_commit(s_full(0));
        if constexpr (TWO) {
          issue_s(1, slot_of(it0));
          mma_commit(s_full(1));
        }
        if (n_kv == 1) mma_commit(q_empty);
        mma_commit(empty_bar(slot_of(it0)));
        if (u_idx > 0 && !mbar_wait(o_free(0), (u_idx - 1) & 1, ab)) return false;
        if constexpr (TWO) {
          if (u2_idx > 0 && !mbar_wait(o_free(1), (u2_idx - 1) & 1, ab)) return false;
        }
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
        const int u = fp8_unit_index(r);
        if (u >= n_units) break;
        const Fp8Unit w = fp8_unit(p, u);
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
      mma_commit(mma_done);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(mma_done, 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_SOFTMAX));
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int w = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + (w ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = tmem + lane_off + (w ? C::COL_O1 : C::COL_O0);
    int jg = 0;
    bool ok = true;
    for (int ru = 0; ok; ++ru) {
      const int u = fp8_unit_index(ru);
      if (u >= n_units) break;
      const Fp8Unit wu = fp8_unit(p, u);
      if (w == 1 && !wu.two) continue;
      const int row = wu.q0 + w * 128 + r;
      const int tile_row0 = wu.q0 + w * 128;
      const int kvh = wu.kv_z;
      // the query tile's block scale times the softmax scale in log2 units
      const float cq = p.scale_log2 * p.sq[(size_t)wu.bh * nb + (tile_row0 >> 7)];
      const float svmax = p.vmax[kvh];
      float m_used = -INFINITY;   // exact running max (log2 units): every growth rescales
      float l_exact = 0.f;        // sum of the unquantised weights
      float l_q = 0.f;            // sum of the quantised weights the PV MMA used
      for (int j = 0; j < wu.n_kv; ++j, ++jg) {
        // this key tile's scales: S in log2 units = s * c, weights 448 f_j p with f_j = sv_j / sv_max
        const float c = cq * p.sk[(size_t)kvh * nb + j];
        const float sv = p.sv[(size_t)kvh * nb + j];
        const float b448 = log2f(448.f * sv / svmax);          // folded into the exponent
        const float inv448f = svmax / (448.f * sv);             // back to unit weights
        ok = __all_sync(0xffffffffu, mbar_wait(s_full(w), jg & 1, ab));
        if (!ok) break;
        tc_fence_after();
        // column cc of the tile is masked from lim on (past N, or after the row when causal),
        // worked out before the row is loaded (as in the bf16 forward: fewer values live)
        const int col0 = j * 128;
        const int lim = p.causal ? min(N - col0, row + 1 - col0) : N - col0;
        const bool mask_tile = (p.causal && col0 + 127 > tile_row0) || col0 + 128 > N;
        float s[128];
        {
          uint32_t rr[128];
          tmem_ld128(tS, rr);
#pragma unroll
          for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(rr[i]);
        }
        if (mask_tile) {
#pragma unroll
          for (int cc = 0; cc < 128; ++cc)
            if (cc >= lim) s[cc] = -INFINITY;
        }
        float mx4[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          float m = fmaxf(s[32 * a], s[32 * a + 1]);
#pragma unroll
          for (int cc = 2; cc < 32; cc += 2) m = max3f(m, s[32 * a + cc], s[32 * a + cc + 1]);
          mx4[a] = m;
        }
        const float m_tile = fmaxf(max3f(mx4[0], mx4[1], mx4[2]), mx4[3]) * c;
        const bool need = m_tile > m_used;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? m_tile : m_used;
          const float alpha = need ? ex2_mufu(m_used - m_new) : 1.f;
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            ok = __all_sync(0xffffffffu, mbar_wait(o_bar(w), (jg - 1) & 1, ab));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              uint32_t rr[16];
              tmem_ld16(tO + 16 * cc, rr);
#pragma unroll
              for (int i = 0; i < 16; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
              tmem_st16(tO + 16 * cc, rr);
            }
            tmem_st_wait();
          }
          l_exact *= alpha;
          l_q *= alpha;
          m_used = m_new;
        }
        const float off = (m_used == -INFINITY) ? 0.f : b448 - m_used;
        const uint64_t c2 = f2_pack(c, c), o2 = f2_pack(off, off);
        uint64_t lsum = 0;     // this tile's sum of 448 f_j p (fp32 pair)
        uint32_t qsum[2] = {0u, 0u};  // this tile's sum of the e4m3 weights (f16 pairs)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int k = 64 * cc + 4 * i;
            const float2 xa = f2_unpack(f2_fma(f2_pack(s[k], s[k + 1]), c2, o2));
            const float2 xb = f2_unpack(f2_fma(f2_pack(s[k + 2], s[k + 3]), c2, o2));
            const float p0 = ex2_mufu(xa.x), p1 = ex2_mufu(xa.y), p2 = ex2_mufu(xb.x), p3 = ex2_mufu(xb.y);
            lsum = f2_add(lsum, f2_add(f2_pack(p0, p1), f2_pack(p2, p3)));
            const uint16_t e01 = pack_e4m3x2(p0, p1), e23 = pack_e4m3x2(p2, p3);
            pk[i] = static_cast<uint32_t>(e01) | (static_cast<uint32_t>(e23) << 16);
            qsum[i & 1] = hadd2(qsum[i & 1], hadd2(e4m3x2_to_f16x2(e01), e4m3x2_to_f16x2(e23)));
          }
          tmem_st16(tS + 16 * cc, pk);
        }
        const float2 ls = f2_unpack(lsum);
        l_exact += (ls.x + ls.y) * inv448f;
        l_q += (f16x2_sum(qsum[0]) + f16x2_sum(qsum[1])) * inv448f;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full(w));
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(o_bar(w), (jg - 1) & 1, ab));
      if (!ok) break;
      tc_fence_after();
      const float inv_l = l_q > 0.f ? svmax / (448.f * l_q) : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + ((size_t)wu.bh * N + row) * 128);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t rr[32];
        tmem_ld32(tO + 32 * cc, rr);
        if (cc == 3) {
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
            orow[cc * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
      if (row < N) p.lse[(size_t)wu.bh * N + row] = l_exact > 0.f ? (m_used + log2f(l_exact)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_fp8_quantize(const void* x, void* out, float* scales, const float* signs, float inv_sqrt_d,
                                long long heads, int N, bool rotate, bool transpose, int pitch, cudaStream_t stream) {
  const int nb = (N + 127) / 128;
  const long long blocks = heads * nb;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)blocks);
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint8_t* o = static_cast<uint8_t*>(out);
  if (transpose)
    fp8_quant_kernel<false, true><<<grid, 256, 0, stream>>>(xs, o, scales, signs, inv_sqrt_d, N, nb, pitch);
  else if (rotate)
    fp8_quant_kernel<true, false><<<grid, 256, 0, stream>>>(xs, o, scales, signs, inv_sqrt_d, N, nb, pitch);
  else
    fp8_quant_kernel<false, false><<<grid, 256, 0, stream>>>(xs, o, scales, signs, inv_sqrt_d, N, nb, pitch);
  return cudaGetLastError();
}

cudaError_t launch_fp8_vmax(const float* sv, float* vmax, long long heads, int N, cudaStream_t stream) {
  const int nb = (N + 127) / 128;
  fp8_vmax_kernel<<<(unsigned)((heads + 7) / 8), 256, 0, stream>>>(sv, vmax, heads, nb);
  return cudaGetLastError();
}

static int fp8_sm_count() {
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

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const Fp8Params& p,
                           cudaStream_t stream) {
  using C = Fp8Cfg;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_done[dev]) {
    e = cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const long long units = (long long)((p.N + 255) / 256) * p.B * p.H;
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(units, fp8_sm_count());
  fwd_fp8_kernel<<<dim3((unsigned)grid), dim3(C::THREADS), C::SMEM_BYTES, stream>>>(tq, tk, tvt, p, (int)units);
  return cudaGetLastError();
}

}  // namespace fa
