// fa_api.cu -- the C ABI declared in include/fa.h: argument validation, tensor
// maps, the device status word and the kernel launches.  All validation runs
// before any CUDA call, so a rejected call never touches the GPU.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {

// The library's device status word (one per device that loads the library).
__device__ int g_status_word;
// Number of O rescales the forward performed while counting was switched on (option
// "count_rescales"); read with fa_get_option("rescale_events"), cleared by setting it to 0.
__device__ unsigned long long g_rescale_events;
// Kernel-wide abort word: a launch whose CTA gives up a wait stores its generation here so the
// launch's other CTAs stop waiting too (see Abort in sm103.cuh).
__device__ unsigned g_abort_word;

// Text of the last FA_ERR_CUDA cause on this host thread.
static thread_local char g_detail[256] = "";

static int cuda_fail(const char* what, cudaError_t e) {
  snprintf(g_detail, sizeof(g_detail), "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
  return FA_ERR_CUDA;
}
static int fail_detail(int status, const char* what) {
  snprintf(g_detail, sizeof(g_detail), "%s", what);
  return status;
}

Options& options() {
  static Options o;
  return o;
}

int* device_status_ptr() {
  static int* ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { cuda_fail("cudaGetDevice", e); return nullptr; }
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) { cuda_fail("cudaGetSymbolAddress(status word)", e); return nullptr; }
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

unsigned long long* rescale_events_ptr() {
  static unsigned long long* ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { cuda_fail("cudaGetDevice", e); return nullptr; }
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_rescale_events);
    if (e != cudaSuccess) { cuda_fail("cudaGetSymbolAddress(rescale events)", e); return nullptr; }
    ptrs[dev] = static_cast<unsigned long long*>(p);
  }
  return ptrs[dev];
}

unsigned* abort_word_ptr() {
  static unsigned* ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { cuda_fail("cudaGetDevice", e); return nullptr; }
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_abort_word);
    if (e != cudaSuccess) { cuda_fail("cudaGetSymbolAddress(abort word)", e); return nullptr; }
    ptrs[dev] = static_cast<unsigned*>(p);
  }
  return ptrs[dev];
}

unsigned next_generation() {
  static std::atomic<unsigned> g{0};
  unsigned v = ++g;
  if (v == 0) v = ++g;  // 0 is the word's initial value: never a launch's generation
  return v;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cuda_fail("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", e);
  });
  return fn;
}

int make_tmap_bf16_rows(CUtensorMap* map, const void* base, int d, long long rows, long long outer, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return -1;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_detail, sizeof(g_detail), "cuTensorMapEncodeTiled: CUresult %d", (int)r);
    return -1;
  }
  return 0;
}

int make_tmap_u8(CUtensorMap* map, const void* base, long long inner, long long pitch, long long rows,
                 long long outer) {
  auto fn = encode_fn();
  if (!fn) return -1;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)pitch, (cuuint64_t)(pitch * rows)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_detail, sizeof(g_detail), "cuTensorMapEncodeTiled (uint8): CUresult %d", (int)r);
    return -1;
  }
  return 0;
}

// sm_103 check, cached per device.
static int check_device() {
  static int state[64] = {};  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= 64) return fail_detail(FA_ERR_UNSUPPORTED, "device ordinal >= 64");
  if (state[dev] == 0) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail("cudaDeviceGetAttribute", e);
    state[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return state[dev] == 1 ? FA_OK : fail_detail(FA_ERR_UNSUPPORTED, "not an sm_103 device");
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape checks common to every entry point.
static int check_shape(int B, int H, int Hkv, int N, int d) {
  if (B < 0 || H < 1 || Hkv < 1 || N < 0) return FA_ERR_INVALID_ARG;
  if (H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H > (1LL << 30) || N > (1 << 30)) return FA_ERR_INVALID_ARG;
  if ((long long)B * H * ((N + 255) / 256) > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

static int check_scale(float scale) { return (std::isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_INVALID_ARG; }

// multiprocessors of the current device (148 if it cannot be read)
static int sm_count_api() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      v <= 0)
    return 148;
  return v;
}

}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

const char* fa_last_error_detail(void) { return g_detail; }

const char* fa_status_string(int s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_MISALIGNED: return "misaligned pointer";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int fa_set_option(const char* key, double value) {
  if (!key || !std::isfinite(value)) return FA_ERR_INVALID_ARG;
  if (!std::strcmp(key, "rescale_threshold")) {
    if (value < 0.0 || value > 64.0) return FA_ERR_INVALID_ARG;
    options().rescale_threshold = static_cast<float>(value);
    return FA_OK;
  }
  if (!std::strcmp(key, "poly_exp")) {
    if (value != -1.0 && value != 0.0 && value != 4.0 && value != 8.0 && value != 12.0 && value != 16.0)
      return FA_ERR_INVALID_ARG;
    options().poly_exp = static_cast<int>(value);
    return FA_OK;
  }
  if (!std::strcmp(key, "poly_fraction")) {  // the same split as a fraction of the exponentials
    if (value == -1.0) { options().poly_exp = -1; return FA_OK; }
    const double cols = value * 32.0;
    if (cols != 0.0 && cols != 4.0 && cols != 8.0 && cols != 12.0 && cols != 16.0) return FA_ERR_INVALID_ARG;
    options().poly_exp = static_cast<int>(cols);
    return FA_OK;
  }
  if (!std::strcmp(key, "debug_drop_kv_load")) {
    if (value != 0.0 && value != 1.0) return FA_ERR_INVALID_ARG;
    options().debug_drop_kv_load = static_cast<int>(value);
    return FA_OK;
  }
  if (!std::strcmp(key, "debug_bwd_hook")) {
    if (value != 0.0 && value != 1.0 && value != 2.0) return FA_ERR_INVALID_ARG;
    options().debug_bwd_hook = static_cast<int>(value);
    return FA_OK;
  }
  if (!std::strcmp(key, "count_rescales")) {
    if (value != 0.0 && value != 1.0) return FA_ERR_INVALID_ARG;
    options().count_rescales = static_cast<int>(value);
    return FA_OK;
  }
  if (!std::strcmp(key, "bwd_2cta")) {
    if (value != 0.0 && value != 1.0) return FA_ERR_INVALID_ARG;
    options().bwd_2cta = static_cast<int>(value);
    return FA_OK;
  }
  if (!std::strcmp(key, "fwd_2cta")) {
    if (value != 0.0 && value != 1.0) return FA_ERR_INVALID_ARG;
    options().fwd_2cta = static_cast<int>(value);
    return FA_OK;
  }
  if (!std::strcmp(key, "rescale_events")) {  // only 0: clear the counter (synchronises the device)
    if (value != 0.0) return FA_ERR_INVALID_ARG;
    unsigned long long* p = rescale_events_ptr();
    if (!p) return FA_ERR_CUDA;
    const unsigned long long zero = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    return e == cudaSuccess ? FA_OK : cuda_fail("clearing the rescale-event counter", e);
  }
  return FA_ERR_INVALID_ARG;
}

int fa_get_option(const char* key, double* value) {
  if (!key || !value) return FA_ERR_INVALID_ARG;
  if (!std::strcmp(key, "rescale_threshold")) { *value = options().rescale_threshold; return FA_OK; }
  if (!std::strcmp(key, "poly_exp")) { *value = options().poly_exp; return FA_OK; }
  if (!std::strcmp(key, "poly_fraction")) {
    *value = options().poly_exp < 0 ? -1.0 : options().poly_exp / 32.0;
    return FA_OK;
  }
  if (!std::strcmp(key, "debug_drop_kv_load")) { *value = options().debug_drop_kv_load; return FA_OK; }
  if (!std::strcmp(key, "debug_bwd_hook")) { *value = options().debug_bwd_hook; return FA_OK; }
  if (!std::strcmp(key, "count_rescales")) { *value = options().count_rescales; return FA_OK; }
  if (!std::strcmp(key, "bwd_2cta")) { *value = options().bwd_2cta; return FA_OK; }
  if (!std::strcmp(key, "fwd_2cta")) { *value = options().fwd_2cta; return FA_OK; }
  if (!std::strcmp(key, "rescale_events")) {  // synchronises the device, then reads the counter
    unsigned long long* p = rescale_events_ptr();
    if (!p) return FA_ERR_CUDA;
    unsigned long long v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail("reading the rescale-event counter", e);
    *value = static_cast<double>(v);
    return FA_OK;
  }
  return FA_ERR_INVALID_ARG;
}

int fa_last_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
  int* p = device_status_ptr();
  if (!p) return FA_ERR_CUDA;
  int v = 0;
  if ((e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail("cudaMemcpy", e);
  const int zero = 0;
  if (v != 0 && (e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail("cudaMemcpy", e);
  return v;
}

int fa_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int Nq,
              int Nk, int d, int causal, float scale, void* stream) {
  int st = check_shape(B, H, Hkv, Nq, d);
  if (st) return st;
  if ((st = check_shape(B, H, Hkv, Nk, d))) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((st = check_scale(scale))) return st;
  if (B == 0 || Nq == 0) return FA_OK;
  if (!q || !o || !lse || (Nk > 0 && (!k || !v))) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  if ((st = check_device())) return st;
  if (Nk == 0) {  // no key: O = 0, LSE = -inf
    cudaError_t e = launch_fwd_no_keys(o, lse, (long long)B * H * Nq, d, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : cuda_fail("fa_fwd (no keys) launch", e);
  }

  CUtensorMap tq, tk, tv;
  if (make_tmap_bf16_rows(&tq, q, d, Nq, (long long)B * H) || make_tmap_bf16_rows(&tk, k, d, Nk, (long long)B * Hkv) ||
      make_tmap_bf16_rows(&tv, v, d, Nk, (long long)B * Hkv))
    return FA_ERR_CUDA;
  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.qoff = Nk - Nq;
  p.causal = causal;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.tau = options().rescale_threshold;
  p.drop_it = options().debug_drop_kv_load ? 2 : -1;
  p.splits = 1;
  p.split_tiles = (Nk + 127) / 128;
  p.pos_mod = 0;
  p.status = device_status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.rescale_events = nullptr;
  if (options().count_rescales && !(p.rescale_events = rescale_events_ptr())) return FA_ERR_CUDA;
  if (!(p.kabort = abort_word_ptr())) return FA_ERR_CUDA;
  p.gen = next_generation();
  // the exponential-split ablation is built for d = 64 and 128 only
  const int poly = (d == 256 || options().poly_exp < 0) ? kDefaultPolyCols : options().poly_exp;
  cudaError_t e;
  if (d == 128 && poly == 0 && options().fwd_2cta) {  // CTA pairs (MUFU exponentials)
    CUtensorMap tk64;
    if (make_tmap_bf16_rows(&tk64, k, d, Nk, (long long)B * Hkv, 64)) return FA_ERR_CUDA;
    e = launch_fwd_pair(tq, tk64, tv, p, static_cast<cudaStream_t>(stream));
  } else {
    e = launch_fwd(d, tq, tk, tv, p, poly, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? FA_OK : cuda_fail("fa_fwd launch", e);
}

// Split-KV forward for few queries against many keys (decoding).  The H/Hkv query heads of a
// K/V group are contiguous in q, o and lse, so they are taken as one head of g*Nq rows (query
// row i of head h becomes row (h % g) * Nq + i, at causal position i + Nk - Nq): K and V are
// then read once per group.  The key tiles are split over `splits` CTAs per 256-row block.
static int splitkv_choice(int B, int H, int Hkv, int Nq, int Nk, int d, int splits) {
  const int rows = (H / Hkv) * Nq;
  const int n_kv = (Nk + 127) / 128;
  if (splits <= 0) {
    // one CTA per SM slot at a time: minimise (waves) x (key tiles per CTA + a fixed cost of
    // about two tiles for the CTA's prologue and epilogue).  With more than one split, units of
    // at most 128 rows run in the decoding configuration: 128-row units, two CTAs per SM.
    const long long sms = sm_count_api();
    const bool dec = fwd_decoding_config(d, rows, 2, 0);
    long long best = -1;
    for (int S = 1; S <= std::min(n_kv, 256); ++S) {
      const bool two = dec && S > 1;
      const long long blocks = (long long)B * Hkv * (two ? (rows + 127) / 128 : (rows + 255) / 256);
      const long long slots = sms * (two ? 2 : 1);
      const long long waves = (blocks * S + slots - 1) / slots;
      const long long cost = waves * ((n_kv + S - 1) / S + 2);
      if (best < 0 || cost < best) {
        best = cost;
        splits = S;
      }
    }
  }
  return std::max(1, std::min(splits, std::max(1, n_kv)));
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d, int splits) {
  if (check_shape(B, H, Hkv, Nq, d) || check_shape(B, H, Hkv, Nk, d) || splits < 0 || splits > 4096) return 0;
  const int S = splitkv_choice(B, H, Hkv, Nq, Nk, d, splits);
  if (S == 1) return 0;
  const size_t rows = (size_t)B * H * Nq;
  return ((size_t)S * rows * d * 4 + 255) / 256 * 256 + (size_t)S * rows * 4;
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int Nq,
                   int Nk, int d, int causal, float scale, int splits, void* workspace, size_t workspace_bytes,
                   void* stream) {
  int st = check_shape(B, H, Hkv, Nq, d);
  if (st) return st;
  if ((st = check_shape(B, H, Hkv, Nk, d))) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((st = check_scale(scale))) return st;
  if (splits < 0 || splits > 4096) return FA_ERR_INVALID_ARG;
  if (B == 0 || Nq == 0) return FA_OK;
  if (Nk == 0) return fa_fwd_qk(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, causal, scale, stream);
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  const int g = H / Hkv;
  if ((long long)g * Nq > (1 << 30)) return FA_ERR_INVALID_ARG;
  const int S = splitkv_choice(B, H, Hkv, Nq, Nk, d, splits);
  const size_t need = fa_fwd_splitkv_workspace_bytes(B, H, Hkv, Nq, Nk, d, splits);
  if (S > 1) {
    if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  }
  if ((st = check_device())) return st;
  const int rows = g * Nq;  // per K/V head
  CUtensorMap tq, tk, tv;
  if (make_tmap_bf16_rows(&tq, q, d, rows, (long long)B * Hkv) || make_tmap_bf16_rows(&tk, k, d, Nk, (long long)B * Hkv) ||
      make_tmap_bf16_rows(&tv, v, d, Nk, (long long)B * Hkv))
    return FA_ERR_CUDA;
  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = Hkv;
  p.Hkv = Hkv;
  p.Nq = rows;
  p.Nk = Nk;
  p.qoff = Nk - Nq;
  p.causal = causal;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.tau = options().rescale_threshold;
  p.drop_it = -1;
  p.splits = S;
  const int n_kv = (Nk + 127) / 128;
  p.split_tiles = (n_kv + S - 1) / S;
  p.pos_mod = Nq;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t all_rows = (size_t)B * H * Nq;
  p.o_part = S > 1 ? reinterpret_cast<float*>(ws) : nullptr;
  p.lse_part = S > 1 ? reinterpret_cast<float*>(ws + ((size_t)S * all_rows * d * 4 + 255) / 256 * 256) : nullptr;
  p.status = device_status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.rescale_events = nullptr;
  if (options().count_rescales && !(p.rescale_events = rescale_events_ptr())) return FA_ERR_CUDA;
  if (!(p.kabort = abort_word_ptr())) return FA_ERR_CUDA;
  p.gen = next_generation();
  // the exponential-split ablation is built for d = 64 and 128 only
  const int poly = (d == 256 || options().poly_exp < 0) ? kDefaultPolyCols : options().poly_exp;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_fwd(d, tq, tk, tv, p, poly, s);
  if (e == cudaSuccess && S > 1) e = launch_fwd_combine(d, p.o_part, p.lse_part, o, lse, S, (long long)all_rows, s);
  return e == cudaSuccess ? FA_OK : cuda_fail("fa_fwd_splitkv launch", e);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N, int d,
           int causal, float scale, void* stream) {
  return fa_fwd_qk(q, k, v, o, lse, B, H, Hkv, N, N, d, causal, scale, stream);
}

// Workspace layout, with the query rows of every head padded to Nqp = Nq rounded up to 128:
// [dQ accumulator fp32 B*H*Nqp*d][lse2 fp32 B*H*Nqp][D fp32 B*H*Nqp][counters int32]; the
// deterministic mode's ordering counters: one per 128-row query tile (d = 64, 128), one per
// 64-row query tile and head-dimension half (d = 256).
struct BwdWorkspace {
  size_t off_lse2, off_d, off_cnt, total;
};
static size_t bwd_counter_count(size_t padded_rows, int d) {
  return d == 256 ? padded_rows / 32 : padded_rows / 128;
}
static BwdWorkspace bwd_ws_layout(int B, int H, int Nq, int d, int deterministic) {
  const size_t Np = ((size_t)Nq + 127) / 128 * 128;
  const size_t rows = (size_t)B * H * Np;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  BwdWorkspace w;
  w.off_lse2 = up(rows * d * 4);
  w.off_d = up(w.off_lse2 + rows * 4);
  w.off_cnt = up(w.off_d + rows * 4);
  w.total = w.off_cnt + (deterministic ? up(bwd_counter_count(rows, d) * 4) : 0);
  return w;
}

size_t fa_bwd_qk_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d, int deterministic) {
  if (check_shape(B, H, Hkv, Nq, d) || check_shape(B, H, Hkv, Nk, d)) return 0;
  if (deterministic != 0 && deterministic != 1) return 0;
  return bwd_ws_layout(B, H, Nq, d, deterministic).total;
}

size_t fa_bwd_workspace_bytes(int B, int H, int Hkv, int N, int d, int deterministic) {
  return fa_bwd_qk_workspace_bytes(B, H, Hkv, N, N, d, deterministic);
}

// Checks shared by the backward stages; returns FA_OK when there is work to launch,
// 1 when there is no query row (nothing to do in the stages), or an error status.
static int check_bwd_common(int B, int H, int Hkv, int Nq, int d, int deterministic, const void* ws,
                            size_t ws_bytes) {
  int st = check_shape(B, H, Hkv, Nq, d);
  if (st) return st;
  if (deterministic != 0 && deterministic != 1) return FA_ERR_INVALID_ARG;
  if (B == 0 || Nq == 0) return 1;
  if (!ws) return FA_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return FA_ERR_MISALIGNED;
  if (ws_bytes < bwd_ws_layout(B, H, Nq, d, deterministic).total) return FA_ERR_WORKSPACE;
  return FA_OK;
}

// The stages below assume their arguments were validated.
static int bwd_pre_impl(const void* o, const void* dout, const float* lse, int B, int H, int Nq, int d,
                        int deterministic, void* workspace, void* stream) {
  const BwdWorkspace w = bwd_ws_layout(B, H, Nq, d, deterministic);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const long long heads = (long long)B * H;
  cudaError_t e = launch_bwd_pre(d, o, dout, lse, reinterpret_cast<float*>(ws + w.off_lse2),
                                 reinterpret_cast<float*>(ws + w.off_d), reinterpret_cast<float*>(ws),
                                 deterministic ? reinterpret_cast<int*>(ws + w.off_cnt) : nullptr, heads, Nq,
                                 (long long)bwd_counter_count((size_t)heads * ((Nq + 127) / 128 * 128), d),
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail("fa_bwd_preprocess launch", e);
}

static int bwd_main_impl(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv, int B,
                         int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, int deterministic,
                         void* workspace, void* stream) {
  CUtensorMap tq, tk, tv, tdo;
  if (make_tmap_bf16_rows(&tq, q, d, Nq, (long long)B * H) || make_tmap_bf16_rows(&tk, k, d, Nk, (long long)B * Hkv) ||
      make_tmap_bf16_rows(&tv, v, d, Nk, (long long)B * Hkv) ||
      make_tmap_bf16_rows(&tdo, dout, d, Nq, (long long)B * H))
    return FA_ERR_CUDA;
  const BwdWorkspace w = bwd_ws_layout(B, H, Nq, d, deterministic);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BwdParams p{};
  p.v = v;
  p.dk = dk;
  p.dv = dv;
  p.dq_acc = reinterpret_cast<float*>(ws);
  p.lse2 = reinterpret_cast<const float*>(ws + w.off_lse2);
  p.dvec = reinterpret_cast<const float*>(ws + w.off_d);
  p.counters = deterministic ? reinterpret_cast<int*>(ws + w.off_cnt) : nullptr;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.qoff = Nk - Nq;
  p.causal = causal;
  p.deterministic = deterministic;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.scale = scale;
  p.status = device_status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.debug_hook = options().debug_bwd_hook;
  if (!(p.kabort = abort_word_ptr())) return FA_ERR_CUDA;
  p.gen = next_generation();
  cudaError_t e;
  if (d == 256) {
    // 64-row query tiles (the four 64-column chunks of a row are loaded as separate boxes)
    CUtensorMap tq64, tdo64;
    if (make_tmap_bf16_rows(&tq64, q, d, Nq, (long long)B * H, 64) ||
        make_tmap_bf16_rows(&tdo64, dout, d, Nq, (long long)B * H, 64))
      return FA_ERR_CUDA;
    e = launch_bwd256(tq64, tk, tdo64, p, static_cast<cudaStream_t>(stream));
  } else if (d == 128 && options().bwd_2cta) {
    CUtensorMap tq64, tdo64;
    if (make_tmap_bf16_rows(&tq64, q, d, Nq, (long long)B * H, 64) ||
        make_tmap_bf16_rows(&tdo64, dout, d, Nq, (long long)B * H, 64))
      return FA_ERR_CUDA;
    e = launch_bwd_main_pair(tq, tq64, tk, tv, tdo, tdo64, p, static_cast<cudaStream_t>(stream));
  } else {
    e = launch_bwd_main(d, tq, tk, tv, tdo, p, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? FA_OK : cuda_fail("fa_bwd_main launch", e);
}

static int bwd_post_impl(void* dq, int B, int H, int Nq, int d, void* workspace, void* stream) {
  cudaError_t e = launch_bwd_post(static_cast<const float*>(workspace), dq, (long long)B * H, Nq, d,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail("fa_bwd_postprocess launch", e);
}

int fa_bwd_preprocess(const void* o, const void* dout, const float* lse, int B, int H, int Hkv, int N, int d,
                      int deterministic, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_bwd_common(B, H, Hkv, N, d, deterministic, workspace, workspace_bytes);
  if (st == 1) return FA_OK;
  if (st) return st;
  if (!o || !dout || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(o, 16) || !aligned(dout, 16) || !aligned(lse, 4)) return FA_ERR_MISALIGNED;
  if ((st = check_device())) return st;
  return bwd_pre_impl(o, dout, lse, B, H, N, d, deterministic, workspace, stream);
}

int fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, const float* lse, void* dk, void* dv,
                int B, int H, int Hkv, int N, int d, int causal, float scale, int deterministic, void* workspace,
                size_t workspace_bytes, void* stream) {
  (void)lse;  // the preprocess stage has staged LSE (in log2 units) into the workspace
  int st = check_bwd_common(B, H, Hkv, N, d, deterministic, workspace, workspace_bytes);
  if (st == 1) return FA_OK;
  if (st) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((st = check_scale(scale))) return st;
  if (!q || !k || !v || !dout || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dout, 16) || !aligned(dk, 16) ||
      !aligned(dv, 16))
    return FA_ERR_MISALIGNED;
  if ((st = check_device())) return st;
  return bwd_main_impl(q, k, v, dout, dk, dv, B, H, Hkv, N, N, d, causal, scale, deterministic, workspace, stream);
}

int fa_bwd_postprocess(void* dq, int B, int H, int Hkv, int N, int d, int deterministic, void* workspace,
                       size_t workspace_bytes, void* stream) {
  int st = check_bwd_common(B, H, Hkv, N, d, deterministic, workspace, workspace_bytes);
  if (st == 1) return FA_OK;
  if (st) return st;
  if (!dq) return FA_ERR_INVALID_ARG;
  if (!aligned(dq, 16)) return FA_ERR_MISALIGNED;
  if ((st = check_device())) return st;
  return bwd_post_impl(dq, B, H, N, d, workspace, stream);
}

}  // extern "C"

namespace fa {

// Every check fa_bwd_qk makes, in its order (shapes, options, workspace, pointers, device).
// Returns FA_OK with *launch set when kernels must run, FA_OK with *launch clear when there is
// nothing to do (B = 0, or no query row and no key), or the error status.
int bwd_validate(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 const void* dq, const void* dk, const void* dv, int B, int H, int Hkv, int Nq, int Nk, int d,
                 int causal, float scale, int deterministic, const void* workspace, size_t workspace_bytes,
                 bool* launch) {
  *launch = false;
  int st = check_shape(B, H, Hkv, Nk, d);
  if (st) return st;
  st = check_bwd_common(B, H, Hkv, Nq, d, deterministic, workspace, workspace_bytes);
  if (st < 0) return st;
  const bool no_queries = st == 1;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((st = check_scale(scale))) return st;
  if (B == 0 || (no_queries && Nk == 0)) return FA_OK;
  if (!no_queries && (!q || !o || !dout || !lse || !dq)) return FA_ERR_INVALID_ARG;
  if (Nk > 0 && (!k || !v || !dk || !dv)) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  if ((st = check_device())) return st;
  *launch = true;
  return FA_OK;
}

int report_cuda_error(const char* what, cudaError_t e) { return cuda_fail(what, e); }

}  // namespace fa

extern "C" {

int fa_bwd_qk(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
              void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq, int Nk, int d, int causal, float scale,
              int deterministic, void* workspace, size_t workspace_bytes, void* stream) {
  // validate everything before the first launch
  bool launch = false;
  int st = bwd_validate(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, Nq, Nk, d, causal, scale, deterministic,
                        workspace, workspace_bytes, &launch);
  if (st || !launch) return st;
  const bool no_queries = Nq == 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (no_queries || Nk == 0) {
    // no query row sees a key: the gradients that exist are zero
    cudaError_t e = cudaSuccess;
    if (no_queries) {
      const size_t kv_bytes = (size_t)B * Hkv * Nk * d * 2;
      e = cudaMemsetAsync(dk, 0, kv_bytes, s);
      if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kv_bytes, s);
    } else {
      e = cudaMemsetAsync(dq, 0, (size_t)B * H * Nq * d * 2, s);
    }
    return e == cudaSuccess ? FA_OK : cuda_fail("cudaMemsetAsync", e);
  }
  st = bwd_pre_impl(o, dout, lse, B, H, Nq, d, deterministic, workspace, stream);
  if (st) return st;
  st = bwd_main_impl(q, k, v, dout, dk, dv, B, H, Hkv, Nq, Nk, d, causal, scale, deterministic, workspace, stream);
  if (st) return st;
  return bwd_post_impl(dq, B, H, Nq, d, workspace, stream);
}

// FP8 workspace layout (each part 256-byte aligned), nb = ceil(N / 128), Np = N rounded up to
// 16: q8 [B*H][N][128], k8 [B*Hkv][N][128], v8t [B*Hkv][128][Np] (e4m3 codes), then fp32 sq
// [B*H][nb], sk [B*Hkv][nb], sv [B*Hkv][nb], vmax [B*Hkv].
static int fp8_layout(int B, int H, int Hkv, int N, size_t off[8]) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t nb = (size_t)(N + 127) / 128, Np = ((size_t)N + 15) / 16 * 16;
  off[0] = 0;
  off[1] = up(off[0] + (size_t)B * H * N * 128);
  off[2] = up(off[1] + (size_t)B * Hkv * N * 128);
  off[3] = up(off[2] + (size_t)B * Hkv * 128 * Np);
  off[4] = up(off[3] + (size_t)B * H * nb * 4);
  off[5] = up(off[4] + (size_t)B * Hkv * nb * 4);
  off[6] = up(off[5] + (size_t)B * Hkv * nb * 4);
  off[7] = up(off[6] + (size_t)B * Hkv * 4);  // total
  return 0;
}

static int check_fp8_shape(int B, int H, int Hkv, int N, int d) {
  int st = check_shape(B, H, Hkv, N, d);
  if (st) return st;
  if (d != 128) return fail_detail(FA_ERR_UNSUPPORTED, "the FP8 forward supports d = 128");
  return FA_OK;
}

size_t fa_fp8_workspace_bytes(int B, int H, int Hkv, int N, int d) {
  if (check_fp8_shape(B, H, Hkv, N, d)) return 0;
  size_t off[8];
  fp8_layout(B, H, Hkv, N, off);
  return off[7];
}

int fa_fp8_workspace_layout(int B, int H, int Hkv, int N, int d, size_t* offsets) {
  int st = check_fp8_shape(B, H, Hkv, N, d);
  if (st) return st;
  if (!offsets) return FA_ERR_INVALID_ARG;
  fp8_layout(B, H, Hkv, N, offsets);
  return FA_OK;
}

int fa_fp8_quantize(const void* q, const void* k, const void* v, const float* signs, int B, int H, int Hkv, int N,
                    int d, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_fp8_shape(B, H, Hkv, N, d);
  if (st) return st;
  if (B == 0 || N == 0) return FA_OK;
  size_t off[8];
  fp8_layout(B, H, Hkv, N, off);
  if (!q || !k || !v) return FA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < off[7]) return FA_ERR_WORKSPACE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(signs, 4) || !aligned(workspace, 256))
    return FA_ERR_MISALIGNED;
  if ((st = check_device())) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float c = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  const int Np = (N + 15) / 16 * 16;
  const bool rot = signs != nullptr;
  cudaError_t e = launch_fp8_quantize(q, ws + off[0], reinterpret_cast<float*>(ws + off[3]), signs, c,
                                      (long long)B * H, N, rot, false, 0, s);
  if (e == cudaSuccess)
    e = launch_fp8_quantize(k, ws + off[1], reinterpret_cast<float*>(ws + off[4]), signs, c, (long long)B * Hkv, N,
                            rot, false, 0, s);
  if (e == cudaSuccess)
    e = launch_fp8_quantize(v, ws + off[2], reinterpret_cast<float*>(ws + off[5]), nullptr, c, (long long)B * Hkv, N,
                            false, true, Np, s);
  if (e == cudaSuccess)
    e = launch_fp8_vmax(reinterpret_cast<const float*>(ws + off[5]), reinterpret_cast<float*>(ws + off[6]),
                        (long long)B * Hkv, N, s);
  return e == cudaSuccess ? FA_OK : cuda_fail("fa_fp8_quantize launch", e);
}

int fa_fwd_fp8(const void* workspace, size_t workspace_bytes, void* o, float* lse, int B, int H, int Hkv, int N, int d,
               int causal, float scale, void* stream) {
  int st = check_fp8_shape(B, H, Hkv, N, d);
  if (st) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((st = check_scale(scale))) return st;
  if (B == 0 || N == 0) return FA_OK;
  size_t off[8];
  fp8_layout(B, H, Hkv, N, off);
  if (!o || !lse) return FA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < off[7]) return FA_ERR_WORKSPACE;
  if (!aligned(o, 16) || !aligned(lse, 4) || !aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  if ((st = check_device())) return st;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  const int Np = (N + 15) / 16 * 16;
  CUtensorMap tq, tk, tvt;
  if (make_tmap_u8(&tq, ws + off[0], 128, 128, N, (long long)B * H) ||
      make_tmap_u8(&tk, ws + off[1], 128, 128, N, (long long)B * Hkv) ||
      make_tmap_u8(&tvt, ws + off[2], Np, Np, 128, (long long)B * Hkv))
    return FA_ERR_CUDA;
  Fp8Params p{};
  p.o = o;
  p.lse = lse;
  p.sq = reinterpret_cast<const float*>(ws + off[3]);
  p.sk = reinterpret_cast<const float*>(ws + off[4]);
  p.sv = reinterpret_cast<const float*>(ws + off[5]);
  p.vmax = reinterpret_cast<const float*>(ws + off[6]);
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = N;
  p.causal = causal;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.status = device_status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  if (!(p.kabort = abort_word_ptr())) return FA_ERR_CUDA;
  p.gen = next_generation();
  cudaError_t e = launch_fwd_fp8(tq, tk, tvt, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail("fa_fwd_fp8 launch", e);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, int B, int H, int Hkv, int N, int d, int causal, float scale, int deterministic,
           void* workspace, size_t workspace_bytes, void* stream) {
  return fa_bwd_qk(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, N, d, causal, scale, deterministic, workspace,
                   workspace_bytes, stream);
}

}  // extern "C"
