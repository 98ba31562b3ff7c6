/*
 * fa.h -- C ABI of the GB300 (sm_103a) IO-aware exact attention library.
 *
 * What it computes.  Exact scaled-dot-product attention, not an approximation
 * ("FlashAttention" wiki note, notes.yuuk.io, section 定義): for every batch b,
 * query head h and query row i, with K/V head g = h / (H / Hkv),
 *
 *     S_ij  = scale * <q_i, k_j>,  S_ij = -inf for j > i when causal
 *     P_ij  = exp(S_ij - LSE_i),   LSE_i = log sum_j exp(S_ij)
 *     O_i   = sum_j P_ij v_j
 *
 * The forward never stores the N x N matrix S or P in device memory: it tiles
 * Q/K/V through on-chip memory with an online softmax (section 定義 item (1);
 * the tiling and online-softmax paragraphs of the singularity-lens.com
 * explainer).  The backward recomputes P from the saved LSE on chip (定義
 * item (2); the explainer's recomputation paragraph) and returns the gradients
 * of L = sum(O * dO):
 *
 *     dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P * (dP - D),
 *     dQ = scale * dS K,  dK = scale * dS^T Q   (dK, dV summed over the query
 *     heads that share a K/V head).
 *
 * Layouts (row-major, contiguous, no padding):
 *     q, o, dout, dq   bf16  [B][H][N][d]
 *     k, v, dk, dv     bf16  [B][Hkv][N][d]
 *     lse              fp32  [B][H][N], natural logarithm
 * Causal masking is top-left aligned (query i sees keys 0..i).
 *
 * Ownership.  The caller allocates every buffer on the current CUDA device,
 * including the backward workspace (size from fa_bwd_workspace_bytes).  The
 * library allocates no device memory and keeps no pointer after a call.
 *
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy default
 * stream).  Calls enqueue work and return; they do not synchronise.
 *
 * Device state.  The library keeps a few words of device memory per device
 * (status word, event counter, the fa_bwd_noalloc scratch) and caches their
 * addresses in the device's primary context on first use: calling
 * cudaDeviceReset while the library is loaded is not supported.
 *
 * Errors.  Every argument is validated before anything is launched, so a call
 * that returns FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_MISALIGNED or
 * FA_ERR_WORKSPACE has not touched the GPU.  FA_ERR_CUDA reports a launch or
 * driver error (cudaGetLastError is left as CUDA set it).  A device-side wait
 * that gives up (bounded at about 2 s) records FA_ERR_DEVICE_TIMEOUT in a
 * device status word, read and cleared by fa_last_device_status.
 *
 * Supported: d in {64, 128, 256} (the FP8 forward: d = 128); H % Hkv == 0;
 * 16-byte aligned bf16 pointers, 4-byte aligned lse; any N >= 0; scale finite
 * and > 0; an sm_103 device.  At d = 256 the backward's main stage runs two
 * CTAs per 128-key tile, one per head-dimension half (a tile's dK and dV
 * accumulators would otherwise fill tensor memory), on 64-row query tiles.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1,     /* null pointer, bad size, H % Hkv != 0, bad scale */
  FA_ERR_UNSUPPORTED = -2,     /* d not supported, not an sm_103 device */
  FA_ERR_MISALIGNED = -3,      /* a pointer is not aligned as required */
  FA_ERR_WORKSPACE = -4,       /* workspace missing or smaller than fa_bwd_workspace_bytes */
  FA_ERR_CUDA = -5,            /* a CUDA runtime/driver call or a launch failed */
  FA_ERR_DEVICE_TIMEOUT = -6   /* a bounded device-side wait gave up */
} fa_status;

/* Forward: o = softmax(scale * q k^T [causal mask]) v, lse = row logsumexp.
 * Inputs q [B,H,N,d], k/v [B,Hkv,N,d] bf16; outputs o bf16 [B,H,N,d] and
 * lse fp32 [B,H,N].  One kernel launch on `stream`. */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int Hkv, int N, int d, int causal, float scale, void* stream);

/* Forward with different query and key lengths: q, o [B,H,Nq,d], lse
 * [B,H,Nq]; k, v [B,Hkv,Nk,d].  causal = 1 aligns the mask bottom-right:
 * query row i sits at position i + (Nk - Nq) and sees keys 0..i + Nk - Nq,
 * so a block of Nq new queries after Nk - Nq cached keys (or one decoding
 * query, Nq = 1) sees every earlier key.  The pages do not treat Nq != Nk;
 * this is the plain reading for a query block that follows earlier keys.  A
 * row that sees no key (Nq > Nk, i < Nq - Nk) gets O = 0 and LSE = -inf, as
 * does every row when Nk = 0.  fa_fwd is fa_fwd_qk with Nq = Nk = N. */
int fa_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, void* stream);

/* Split-KV forward for decoding (few queries, many keys); same inputs,
 * outputs and mask as fa_fwd_qk.  The H/Hkv query heads that share a K/V head
 * are processed together as one block of rows, so K and V are read once per
 * group, and the keys are divided among `splits` CTAs per block (0 = choose:
 * about two CTAs per SM).  Each split writes an fp32 partial O, normalised
 * over its keys, and its LSE into the workspace; a second kernel merges them
 * with the online-softmax rule (the running-max rescaling of the explainer's
 * online-softmax paragraph applied to whole splits): LSE = log sum_s e^LSE_s,
 * O = sum_s e^(LSE_s - LSE) O_s.  The pages describe no decoding kernel; this
 * is the merge of independent partial softmaxes that the online softmax
 * implies.  Workspace: fa_fwd_splitkv_workspace_bytes(...) bytes, 256-byte
 * aligned (0 bytes, and a null workspace allowed, when one split is chosen). */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d, int splits);
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, int splits,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace fa_bwd needs, with the rows of every head padded
 * to Np = N rounded up to a multiple of 128: the fp32 dQ accumulator
 * [B,H,Np,d], one (LSE in log2 units, D) fp32 pair per padded query row, and
 * (deterministic mode) one int32 ordering counter per (b, h, 128-row query
 * block), at d = 256 per (b, h, 64-row query block, head-dimension half).
 * The workspace must be 256-byte aligned.  0 on bad sizes. */
size_t fa_bwd_workspace_bytes(int B, int H, int Hkv, int N, int d, int deterministic);

/* Backward: dq, dk, dv (bf16) from q, k, v, o, dout (bf16) and lse (fp32, as
 * written by fa_fwd).  deterministic = 1 makes the dQ accumulation order fixed
 * so repeated calls give bit-identical results (FA4's deterministic backward
 * mode, named in the wiki's 未解決の問い section).  Runs fa_bwd_preprocess,
 * fa_bwd_main and fa_bwd_postprocess on `stream`. */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv,
           int B, int H, int Hkv, int N, int d, int causal, float scale, int deterministic,
           void* workspace, size_t workspace_bytes, void* stream);

/* Backward with different query and key lengths (the mask of fa_fwd_qk):
 * q, o, dout, dq [B,H,Nq,d], lse [B,H,Nq]; k, v, dk, dv [B,Hkv,Nk,d].  Rows
 * that see no key get dQ = 0 and add nothing to dK, dV; keys no query sees
 * get dK = dV = 0.  The workspace (256-byte aligned) must hold
 * fa_bwd_qk_workspace_bytes(...) bytes; its size depends on Nq only.
 * fa_bwd is fa_bwd_qk with Nq = Nk = N. */
size_t fa_bwd_qk_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d, int deterministic);
int fa_bwd_qk(const void* q, const void* k, const void* v, const void* o, const void* dout,
              const float* lse, void* dq, void* dk, void* dv,
              int B, int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, int deterministic,
              void* workspace, size_t workspace_bytes, void* stream);

/* The three stages of fa_bwd, exposed so that callers (and the benchmark) can
 * time or schedule them separately; they must run in this order on one
 * stream with the same workspace.  Same argument checks as fa_bwd.
 *   preprocess : D_i = sum_c dO_ic O_ic (fp32) and LSE_i * log2(e) into the
 *                workspace; zero the dQ accumulator (and counters)
 *   main       : recompute P from LSE tile by tile; write dK, dV; accumulate
 *                scale * dS K into the dQ accumulator.  `lse` is accepted for
 *                symmetry and not read (preprocess staged it).
 *   postprocess: dQ = accumulator rounded to bf16 */
int fa_bwd_preprocess(const void* o, const void* dout, const float* lse, int B, int H, int Hkv, int N,
                      int d, int deterministic, void* workspace, size_t workspace_bytes, void* stream);
int fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, const float* lse,
                void* dk, void* dv, int B, int H, int Hkv, int N, int d, int causal, float scale,
                int deterministic, void* workspace, size_t workspace_bytes, void* stream);
int fa_bwd_postprocess(void* dq, int B, int H, int Hkv, int N, int d,
                       int deterministic, void* workspace, size_t workspace_bytes, void* stream);

/* FP8 (e4m3) forward, head dimension 128: block quantisation with incoherent
 * processing ("FlashAttention" wiki note, section FA3 item 3).  Two calls:
 *
 * fa_fp8_quantize writes the quantised inputs into a caller workspace of
 * fa_fp8_workspace_bytes(...) bytes (256-byte aligned).  q [B,H,N,128], k, v
 * [B,Hkv,N,128] bf16.  If `signs` (device memory, 128 floats, each +1 or -1)
 * is not NULL, every row of Q and K is first rotated by H diag(signs)/sqrt(128),
 * H the Sylvester Hadamard matrix (a fast Walsh-Hadamard transform in fp32),
 * which leaves Q K^T unchanged; the random signs are the caller's.  Each block
 * of 128 rows of one head gets one scale, amax / 448, and the codes
 * e4m3(x * 448 / amax) (round to nearest even, saturating).  Workspace layout
 * (byte offsets from fa_fp8_workspace_layout, 8 values, the last the total):
 * q8 [B*H][N][128], k8 [B*Hkv][N][128], v8 transposed [B*Hkv][128][Np] (Np = N
 * rounded up to 16, padding zero), then fp32 block scales sq [B*H][nb],
 * sk [B*Hkv][nb], sv [B*Hkv][nb] (nb = ceil(N/128)) and vmax [B*Hkv] (the
 * largest V block scale of each K/V head).
 *
 * fa_fwd_fp8 computes attention from that workspace: S from the codes with
 * fp32 accumulation and the block scales, an exact running max, the weights
 * quantised to e4m3 (448 * (sv_block / vmax) * p, the V block scale folded in),
 * O normalised by the sum of the quantised weights, LSE from the unquantised
 * sum.  Outputs o bf16 [B,H,N,128], lse fp32 [B,H,N] (natural log); causal masks
 * are top-left aligned.  The pages give no formats, block sizes or matrices:
 * these are this library's readings (e4m3, 128-row blocks, amax/448 scales). */
size_t fa_fp8_workspace_bytes(int B, int H, int Hkv, int N, int d);
int fa_fp8_workspace_layout(int B, int H, int Hkv, int N, int d, size_t* offsets);
int fa_fp8_quantize(const void* q, const void* k, const void* v, const float* signs,
                    int B, int H, int Hkv, int N, int d, void* workspace, size_t workspace_bytes,
                    void* stream);
int fa_fwd_fp8(const void* workspace, size_t workspace_bytes, void* o, float* lse,
               int B, int H, int Hkv, int N, int d, int causal, float scale, void* stream);

/* Size of the scratch array that fa_bwd_noalloc uses (32 MiB per device). */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)

/* fa_bwd_noalloc -- the backward for callers that cannot allocate device
 * memory.  (The paper has no counterpart: this is a convenience of this
 * library.)  fa_bwd needs a caller-allocated workspace; some callers have no
 * allocator at the call site -- e.g. a plugin or operator run by a host
 * framework that owns all device memory and hands out no scratch, or code on a
 * latency-critical path where cudaMalloc is not allowed because it can
 * synchronise the device.  This entry point takes the same inputs and outputs
 * as fa_bwd (the caller still owns q, k, v, o, dout, lse, dq, dk, dv) but uses
 * a fixed, library-owned device array of FA_NOALLOC_SCRATCH_BYTES as its
 * workspace, and allocates nothing.
 *   - A problem with fa_bwd_workspace_bytes(...) > FA_NOALLOC_SCRATCH_BYTES is
 *     rejected with FA_ERR_WORKSPACE before anything runs.
 *   - Each device that loads the library holds the array until process exit.
 *   - All calls share the array; it keeps the last call's contents, and the
 *     call itself clears what must start at zero.  Calls that may overlap on
 *     the GPU (several streams or host threads on one device) race on it:
 *     serialise them on one stream.
 *   - The first call on a device looks up the array's device address and
 *     caches it; make that first call before any stream capture.
 * Other arguments, checks (in the same order) and status codes are those of
 * fa_bwd, the scratch taking the workspace's place: FA_ERR_WORKSPACE means
 * the problem needs more than FA_NOALLOC_SCRATCH_BYTES. */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv,
                   int B, int H, int Hkv, int N, int d, int causal, float scale, int deterministic,
                   void* stream);

/* Ablation switches (process-wide; take effect on the next call):
 *   "rescale_threshold"  tau >= 0 in log2 units (default 8): the running-max
 *                        correction of O and l is skipped unless the row max
 *                        grew by more than tau (FA4 conditional rescaling,
 *                        ai-papers.net summary, 提案手法 item 2).  0 rescales
 *                        whenever the max grows.
 *   "poly_exp"           exp2 split between the MUFU unit and an FMA-pipe
 *                        polynomial (wiki FA4 (2)) in the forward: number of
 *                        columns out of every 32 computed by the polynomial,
 *                        one of 0, 4, 8, 12, 16; -1 = the built-in default.
 *   "poly_fraction"      the same split as a fraction of the exponentials:
 *                        0, 0.125, 0.25, 0.375 or 0.5; -1 = the default.
 *   "count_rescales"     0 (default) or 1: the forward counts, in a device
 *                        counter, every (row, key tile) at which it rescaled O
 *                        (a debug aid that shows the conditional rescale
 *                        firing or being skipped; one atomic per warp and
 *                        rescale when on, nothing when off).
 *   "rescale_events"     the counter: fa_get_option synchronises the device and
 *                        reads it; fa_set_option(.., 0) synchronises and clears
 *                        it (any other value is rejected).
 *   "bwd_2cta"           1: the backward's main stage runs on CTA pairs (tcgen05
 *                        cta_group::2 MMAs over 256 keys, dS exchanged through
 *                        distributed shared memory), d = 128; 0 (default): one
 *                        CTA per 128-key tile (FA4's two-CTA backward mode, the
 *                        ai-papers.net summary, 提案手法 item 3).
 *   "fwd_2cta"           1: the forward runs on CTA pairs (M = 256 MMAs over 512
 *                        query rows, P in shared memory), d = 128, one split,
 *                        MUFU exponentials; 0: one CTA per 256 query rows.
 *   "debug_drop_kv_load" failure-injection test hook, 0 (default) or 1: the
 *                        forward's copy warp skips its second K/V tile load, so
 *                        the MMA warp's bounded wait gives up (after ~2 s), the
 *                        CTA drains and exits, and fa_last_device_status()
 *                        returns FA_ERR_DEVICE_TIMEOUT.  Output is undefined
 *                        while it is set.
 *   "debug_bwd_hook"     failure-injection test hook of the backward, 0
 *                        (default), 1 (the first CTA, at d = 256 the first
 *                        two, never releases the deterministic mode's ordering
 *                        counters, so the next key tile's bounded spin gives
 *                        up) or 2 (the copy warp skips the second query tile's
 *                        Q/dO load, at d = 256 every load from the second
 *                        tile on, so the MMA warp's bounded wait gives up);
 *                        then as above.
 * Returns FA_OK, FA_ERR_INVALID_ARG (unknown key or value out of range) or,
 * for "rescale_events", FA_ERR_CUDA. */
int fa_set_option(const char* key, double value);
int fa_get_option(const char* key, double* value);

/* Static description of a status code; never NULL. */
const char* fa_status_string(int status);

/* Synchronise `stream`, then return and clear the device status word:
 * FA_OK, or FA_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait since the
 * last call, or FA_ERR_CUDA if the synchronisation itself failed. */
int fa_last_device_status(void* stream);

/* Text describing the cause of the last FA_ERR_CUDA / FA_ERR_UNSUPPORTED
 * returned on the calling host thread (the failing call and CUDA's error
 * string); "" if none.  Owned by the library, valid until the next call. */
const char* fa_last_error_detail(void);

/* Library ABI version (major * 100 + minor). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
