// fa_internal.h -- host-side declarations shared by the C-ABI file and the
// kernel files (launchers and parameter blocks).  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

// Runtime-tunable switches (set through fa_set_option).
struct Options {
  float rescale_threshold = 8.0f;  // tau, log2 units: skip the O/l rescale unless the row max grows by more
  int poly_exp = -1;               // exp2 split: columns of every 32 on the FMA polynomial (0,4,8,12,16; -1 = default)
  int debug_drop_kv_load = 0;      // failure-injection test hook: the forward skips one K/V load
  int debug_bwd_hook = 0;          // failure-injection test hook of the backward: 1 = the first CTA never
                                   // releases its deterministic-order counters, 2 = the copy warp skips
                                   // the second query tile's Q/dO load
  int count_rescales = 0;          // count the forward's O rescales into the library's event counter
  int bwd_2cta = 0;                // backward main stage on CTA pairs (tcgen05 cta_group::2), d = 128
  int fwd_2cta = 0;                // forward on CTA pairs with P in shared memory, d = 128
};
Options& options();

struct FwdParams {
  void* o;           // bf16 [B,H,Nq,d]
  float* lse;        // fp32 [B,H,Nq], natural log
  int B, H, Hkv, Nq, Nk;
  int qoff;          // causal: query row i sits at position i + qoff = i + Nk - Nq
  int causal;
  float scale_log2;  // softmax scale * log2(e)
  float tau;         // rescale threshold, log2 units
  int* status;       // device status word
  int drop_it;       // failure-injection test hook: K/V load index the producer skips (-1: none)
  // split-KV (decode): the key tiles are divided among `splits` CTAs per query block, each
  // writing an fp32 partial O (normalised over its keys) and its LSE (log2 units); a combine
  // kernel merges them.  splits = 1 is the plain forward (bf16 O, natural-log LSE).
  int splits;
  int split_tiles;   // key tiles per split
  int pos_mod;       // causal: row r sits at position (r % pos_mod) + qoff (query heads packed
                     // as rows, pos_mod = Nq); 0: position r + qoff
  float* o_part;     // splits > 1: fp32 [splits][B*H][Nq][d]
  float* lse_part;   // splits > 1: fp32 [splits][B*H][Nq]
  unsigned long long* rescale_events;  // non-null: add the number of rows whose O was rescaled (per key tile)
  unsigned* kabort;  // kernel-wide abort word (see Abort in sm103.cuh)
  unsigned gen;      // this launch's generation
};

struct BwdParams {
  const void* v;      // bf16 [B,Hkv,Nk,d] (read with plain loads by the d = 256 kernel)
  void* dk;           // bf16 [B,Hkv,Nk,d]
  void* dv;           // bf16 [B,Hkv,Nk,d]
  float* dq_acc;      // fp32 [B,H,Nqp,d] dQ accumulator, rows padded to Nqp = Nq rounded up to 128 (workspace)
  const float* lse2;  // per padded query row LSE * log2(e) (workspace)
  const float* dvec;  // per padded query row D = sum_c dO_c O_c (workspace)
  int* counters;      // deterministic mode: ordering counters, [B*H*(Nqp/128)] ([B*H*(Nqp/64)*2] at d = 256)
  int B, H, Hkv, Nq, Nk;
  int qoff;           // causal: query row i sits at position i + qoff = i + Nk - Nq
  int causal;
  int deterministic;
  float scale_log2;   // softmax scale * log2(e)
  float scale;        // softmax scale (folded into dS)
  int* status;        // device status word
  int debug_hook;     // failure-injection test hook (Options::debug_bwd_hook)
  unsigned* kabort;   // kernel-wide abort word (see Abort in sm103.cuh)
  unsigned gen;       // this launch's generation
};

// FP8 forward (fa_fp8.cu), head dimension 128.
struct Fp8Params {
  void* o;              // bf16 [B,H,N,128]
  float* lse;           // fp32 [B,H,N], natural log
  const float* sq;      // block scales [B*H][nb], [B*Hkv][nb] (nb = ceil(N / 128))
  const float* sk;
  const float* sv;
  const float* vmax;    // largest V block scale per K/V head [B*Hkv]
  int B, H, Hkv, N;
  int causal;
  float scale_log2;     // softmax scale * log2(e)
  int* status;
  unsigned* kabort;
  unsigned gen;
};
// Quantise one tensor [heads][N][128] (bf16) to e4m3 codes with one scale per 128-row block;
// rotate: incoherent processing with signs (d floats, +-1, device memory) and 1/sqrt(d);
// transpose: write codes as [heads][128][pitch] (V).
cudaError_t launch_fp8_quantize(const void* x, void* out, float* scales, const float* signs, float inv_sqrt_d,
                                long long heads, int N, bool rotate, bool transpose, int pitch, cudaStream_t stream);
cudaError_t launch_fp8_vmax(const float* sv, float* vmax, long long heads, int N, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const Fp8Params& p,
                           cudaStream_t stream);
// 3-D uint8 tensor map over [outer][rows][inner] bytes (row pitch `pitch` bytes) with a
// 128 x 128 byte box and 128-byte swizzle.  Returns 0 on success.
int make_tmap_u8(CUtensorMap* map, const void* base, long long inner, long long pitch, long long rows,
                 long long outer);

cudaError_t launch_bwd_pre(int d, const void* o, const void* dout, const float* lse, float* lse2, float* dvec,
                           float* dq_acc, int* counters, long long heads, int N, long long n_counters,
                           cudaStream_t stream);
cudaError_t launch_bwd_main(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream);
// The main stage on CTA pairs (d = 128): tq/tdo with 128-row boxes, tq64/tdo64 with 64-row boxes.
cudaError_t launch_bwd_main_pair(const CUtensorMap& tq, const CUtensorMap& tq64, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdo64,
                                 const BwdParams& p, cudaStream_t stream);
// d = 256: two CTAs per key tile, one per head-dimension half (tq64, tdo64: 64-row boxes;
// V is read through p.v)
cudaError_t launch_bwd256(const CUtensorMap& tq64, const CUtensorMap& tk, const CUtensorMap& tdo64,
                          const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_post(const float* dq_acc, void* dq, long long heads, int N, int d, cudaStream_t stream);
// The forward on CTA pairs (d = 128, one split, MUFU exponentials): tq and tv with 128-row
// boxes, tk64 with a 64-row box.
cudaError_t launch_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tk64, const CUtensorMap& tv, const FwdParams& p,
                            cudaStream_t stream);
// Merge split-KV partials: LSE = log sum_s 2^lse_s, O = sum_s 2^(lse_s - LSE) o_s (bf16)
cudaError_t launch_fwd_combine(int d, const float* o_part, const float* lse_part, void* o, float* lse, int splits,
                               long long rows, cudaStream_t stream);
// O = 0 and LSE = -inf for every query row (attention over zero keys)
cudaError_t launch_fwd_no_keys(void* o, float* lse, long long rows, int d, cudaStream_t stream);

// Launch the forward kernel for head dim d (64 or 128) with poly_cols of every 32
// exponentials on the FMA polynomial (0, 4, 8, 12 or 16).  Returns a cudaError_t.
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int poly_cols, cudaStream_t stream);
// Whether launch_fwd takes the decoding configuration (two CTAs per SM, one query tile each):
// split-KV launches (splits > 1) whose units hold at most 128 query rows, MUFU exponentials.
bool fwd_decoding_config(int d, int rows, int splits, int poly_cols);
constexpr int kDefaultPolyCols = 0;

// Build a 3-D bf16 tensor map over a contiguous [outer][rows][d] array with a
// box of 64 x box_rows x 1 elements and 128-byte swizzle.  Returns 0 on success.
int make_tmap_bf16_rows(CUtensorMap* map, const void* base, int d, long long rows, long long outer,
                        int box_rows = 128);

// Device address of the library's status word on the current device (nullptr on error).
int* device_status_ptr();
// Every argument check of fa_bwd_qk, in its order; *launch tells whether kernels must run.
int bwd_validate(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 const void* dq, const void* dk, const void* dv, int B, int H, int Hkv, int Nq, int Nk, int d,
                 int causal, float scale, int deterministic, const void* workspace, size_t workspace_bytes,
                 bool* launch);
// Record `what` and CUDA's error text for fa_last_error_detail; returns FA_ERR_CUDA.
int report_cuda_error(const char* what, cudaError_t e);

// Device address of the library's kernel-wide abort word on the current device (nullptr on
// error), and a fresh non-zero generation for the next launch.
unsigned* abort_word_ptr();
unsigned next_generation();

// Device address of the library's rescale-event counter on the current device (nullptr on error).
unsigned long long* rescale_events_ptr();

}  // namespace fa
