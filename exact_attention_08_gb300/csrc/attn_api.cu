// C ABI of the exact-attention library: argument validation, TMA tensor-map
// construction, device-status word, launches.  See include/attn.h for the
// contract of every entry point.
#include "attn.h"
#include "attn_internal.h"
#include "sm103_ptx.cuh"

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

namespace attn {
namespace {

__device__ int g_attn_status;

thread_local std::string t_last_error;

int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int cuda_error(cudaError_t e, const char* what) {
  return set_error(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- per-device state
constexpr int kMaxDevices = 64;
struct DeviceState {
  bool checked = false;
  bool supported = false;
  int num_sms = 0;
  int* status = nullptr;
};
std::mutex g_dev_mutex;
DeviceState g_dev[kMaxDevices];

// Checks the current device once (sm_103) and resolves the status word.
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return set_error(ATTN_ERR_UNSUPPORTED, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceState& s = g_dev[dev];
  if (!s.checked) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute");
    s.supported = (major == 10 && minor == 3);
    if (s.supported) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_attn_status);
      if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(status)");
      s.status = static_cast<int*>(ptr);
      e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute(SM count)");
    }
    s.checked = true;
    if (!s.supported)
      return set_error(ATTN_ERR_UNSUPPORTED, "device %d is sm_%d%d, this library needs sm_103",
                       dev, major, minor);
  }
  if (!s.supported) return set_error(ATTN_ERR_UNSUPPORTED, "device %d is not sm_103", dev);
  *out = &s;
  return ATTN_OK;
}

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D bf16 tensor (d, n1, n2, n3), innermost first, contiguous; box
// 64 x 1 x box2 x 1 with the 128-byte swizzle.
// s1, s2, s3: strides of dimensions 1..3 in elements (0: contiguous).
int make_map(CUtensorMap* m, const void* ptr, uint64_t d, uint64_t n1, uint64_t n2, uint64_t n3,
             uint32_t box2, const char* what, uint64_t s1 = 0, uint64_t s2 = 0, uint64_t s3 = 0) {
  auto fn = encode_fn();
  if (!fn) return set_error(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[4] = {d, n1, n2, n3};
  if (s1 == 0) s1 = d;
  if (s2 == 0) s2 = n1 * d;
  if (s3 == 0) s3 = n2 * n1 * d;
  cuuint64_t strides[3] = {s1 * 2, s2 * 2, s3 * 2};
  cuuint32_t box[4] = {64, 1, box2, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(ATTN_ERR_INVALID_ARG, "tensor map for %s rejected (CUresult %d)", what,
                     static_cast<int>(r));
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- timeout check
__global__ void wait_timeout_check_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  // Nothing ever arrives on this barrier: the bounded wait must give up.
  const bool ok = ptx::mbar_wait(&bar, 0, nullptr, limit_ns);
  if (!ok && threadIdx.x == 0) atomicOr(status, kStatusTimeout);
}

// ---------------------------------------------------------------- fixed scratch
// Scratch for attn_decode_paged_noalloc: the split partial outputs and
// log-sum-exps live in this array instead of a caller-provided workspace.
// Every device that loads the library holds these 16 MiB until the process
// exits.  Host code must not use the symbol as a pointer: its device address
// is looked up once per device (cudaGetSymbolAddress, with that device
// current) and kept in g_noalloc_scratch_ptr.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
std::mutex g_noalloc_mutex;
void* g_noalloc_scratch_ptr[kMaxDevices];

}  // namespace

cudaError_t launch_wait_timeout_check(int* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_check_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace attn

using namespace attn;

extern "C" {

ATTN_API const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    case ATTN_ERR_BAD_INPUT: return "out-of-range device data (page index or sequence offsets)";
    default: return "unknown status";
  }
}

ATTN_API const char* attn_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"

namespace {

// Every forward entry point: checks, tensor maps, launch.  sink: per-head
// logit sink [Hq] (device, fp32) or null.
// Strides (host arrays of batch, row and head strides in elements, d
// contiguous), null for the contiguous layout; dense calls only.
struct Strides {
  const long long* q = nullptr;
  const long long* k = nullptr;
  const long long* v = nullptr;
  const long long* o = nullptr;
};

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse,
             const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq, int Hkv, int max_Sq,
             int max_Skv, int total_q, int total_k, int d, float scale, int causal, int window,
             int n_sink, const float* sink, void* stream, const Strides& st_in = Strides()) {
  t_last_error.clear();
  const bool varlen = cu_seqlens_q != nullptr || cu_seqlens_k != nullptr;
  if (varlen && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr))
    return set_error(ATTN_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must both be given");
  if (B < 0 || Hq <= 0 || Hkv <= 0 || max_Sq < 0 || max_Skv < 0 || total_q < 0 || total_k < 0)
    return set_error(ATTN_ERR_INVALID_ARG, "negative or zero size (B=%d Hq=%d Hkv=%d)", B, Hq, Hkv);
  if (Hq % Hkv != 0)
    return set_error(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (d != 64 && d != 128 && d != 256)
    return set_error(ATTN_ERR_UNSUPPORTED, "head dim %d (64, 128 or 256)", d);
  if (!(scale > 0.f) || !std::isfinite(scale))
    return set_error(ATTN_ERR_INVALID_ARG, "scale must be finite and positive");
  if (causal != 0 && causal != 1) return set_error(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (window < 0) window = 0;
  if (window > 0 && !causal)
    return set_error(ATTN_ERR_INVALID_ARG, "a sliding window requires causal");
  if (n_sink < 0 || (n_sink > 0 && window == 0))
    return set_error(ATTN_ERR_INVALID_ARG, "n_sink > 0 requires a window");
  const long long rows_q = varlen ? total_q : static_cast<long long>(B) * max_Sq;
  const long long rows_k = varlen ? total_k : static_cast<long long>(B) * max_Skv;
  if (B == 0 || rows_q == 0) return ATTN_OK;
  if (q == nullptr || o == nullptr) return set_error(ATTN_ERR_INVALID_ARG, "q and o must be set");
  if (rows_k > 0 && (k == nullptr || v == nullptr))
    return set_error(ATTN_ERR_INVALID_ARG, "k and v must be set");
  if (!aligned16(q) || !aligned16(o) || !aligned16(k) || !aligned16(v) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(sink) & 3u))
    return set_error(ATTN_ERR_INVALID_ARG,
                     "tensors must be 16-byte aligned (lse and sink 4-byte)");
  if (varlen && max_Sq == 0) return set_error(ATTN_ERR_INVALID_ARG, "max_Sq must bound the lengths");
  // batch, row, head strides of every tensor (elements)
  long long str[4][3];
  {
    const long long* given[4] = {st_in.q, st_in.k, st_in.v, st_in.o};
    const long long H[4] = {Hq, Hkv, Hkv, Hq};
    const long long S[4] = {max_Sq, max_Skv, max_Skv, max_Sq};
    for (int t = 0; t < 4; ++t) {
      if (given[t] == nullptr) {
        str[t][2] = d;
        str[t][1] = H[t] * d;
        str[t][0] = S[t] * H[t] * d;
        continue;
      }
      if (varlen) return set_error(ATTN_ERR_INVALID_ARG, "strides apply to the dense layout only");
      for (int x = 0; x < 3; ++x) {
        str[t][x] = given[t][x];
        if (str[t][x] <= 0 || (str[t][x] % 8) != 0)
          return set_error(ATTN_ERR_INVALID_ARG,
                           "strides must be positive multiples of 8 elements (16 bytes)");
      }
    }
  }

  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != ATTN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  FwdLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.o = o;
  a.lse = lse;
  a.sink = sink;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = max_Sq;
  a.Skv = max_Skv;
  a.total_q = total_q;
  a.total_k = total_k;
  a.d = d;
  a.scale = scale;
  a.causal = causal;
  a.window = window;
  a.n_sink = n_sink;
  a.num_sms = ds->num_sms;
  a.status = ds->status;
  a.o_sb = varlen ? 0 : str[3][0];
  a.o_ss = varlen ? static_cast<long long>(Hq) * d : str[3][1];
  a.o_sh = varlen ? d : str[3][2];
  if (rows_k == 0) {
    cudaError_t e = launch_attn_fill_empty(a, st);
    return e == cudaSuccess ? ATTN_OK : cuda_error(e, "fill launch");
  }
  const uint64_t sq = varlen ? static_cast<uint64_t>(total_q) : static_cast<uint64_t>(max_Sq);
  const uint64_t sk = varlen ? static_cast<uint64_t>(total_k) : static_cast<uint64_t>(max_Skv);
  const uint64_t nb = varlen ? 1u : static_cast<uint64_t>(B);
  if (varlen) {
    if ((rc = make_map(&a.tmQ, q, d, Hq, sq, nb, 128, "q")) != ATTN_OK) return rc;
    if ((rc = make_map(&a.tmK, k, d, Hkv, sk, nb, 128, "k")) != ATTN_OK) return rc;
    if ((rc = make_map(&a.tmV, v, d, Hkv, sk, nb, 128, "v")) != ATTN_OK) return rc;
    if ((rc = make_map(&a.tmO, o, d, Hq, sq, nb, 128, "o")) != ATTN_OK) return rc;
  } else {
    const void* ptr[4] = {q, k, v, o};
    CUtensorMap* map[4] = {&a.tmQ, &a.tmK, &a.tmV, &a.tmO};
    const uint64_t H[4] = {static_cast<uint64_t>(Hq), static_cast<uint64_t>(Hkv),
                           static_cast<uint64_t>(Hkv), static_cast<uint64_t>(Hq)};
    const uint64_t S[4] = {sq, sk, sk, sq};
    const char* nm[4] = {"q", "k", "v", "o"};
    for (int t = 0; t < 4; ++t)
      if ((rc = make_map(map[t], ptr[t], d, H[t], S[t], nb, 128, nm[t], str[t][2], str[t][1],
                         str[t][0])) != ATTN_OK)
        return rc;
  }
  cudaError_t e = launch_attn_fwd(a, st);
  return e == cudaSuccess ? ATTN_OK : cuda_error(e, "attn_fwd launch");
}

}  // namespace

extern "C" {

ATTN_API int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                         const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq, int Hkv,
                         int max_Sq, int max_Skv, int total_q, int total_k, int d, float scale,
                         int causal, int window, int n_sink, void* stream) {
  return fwd_impl(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, max_Sq, max_Skv,
                  total_q, total_k, d, scale, causal, window, n_sink, nullptr, stream);
}

ATTN_API int attn_fwd_ex_sink(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                              int Hkv, int max_Sq, int max_Skv, int total_q, int total_k, int d,
                              float scale, int causal, int window, int n_sink,
                              const float* sink_logit, void* stream) {
  return fwd_impl(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, max_Sq, max_Skv,
                  total_q, total_k, d, scale, causal, window, n_sink, sink_logit, stream);
}

ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int Hq, int Hkv, int Sq, int Skv, int d, float scale, int causal, int window,
                      void* stream) {
  return attn_fwd_ex(q, k, v, o, lse, nullptr, nullptr, B, Hq, Hkv, Sq, Skv, 0, 0, d, scale,
                     causal, window, 0, stream);
}

ATTN_API int attn_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int Sq, int Skv, int d,
                              const long long* q_strides, const long long* k_strides,
                              const long long* v_strides, const long long* o_strides, float scale,
                              int causal, int window, int n_sink, const float* sink_logit,
                              void* stream) {
  Strides st;
  st.q = q_strides;
  st.k = k_strides;
  st.v = v_strides;
  st.o = o_strides;
  return fwd_impl(q, k, v, o, lse, nullptr, nullptr, B, Hq, Hkv, Sq, Skv, 0, 0, d, scale, causal,
                  window, n_sink, sink_logit, stream, st);
}

ATTN_API int attn_fwd_paged(const void* q, const void* k_pages, const void* v_pages,
                            const int* page_table, const int* cu_seqlens_q, const int* seqlens_k,
                            void* o, float* lse, int B, int Hq, int Hkv, int max_Sq, int total_q,
                            int d, int page_size, int max_pages_per_seq, int num_pages_total,
                            float scale, int causal, int window, int n_sink,
                            const float* sink_logit, void* stream) {
  t_last_error.clear();
  if (B < 0 || Hq <= 0 || Hkv <= 0 || max_Sq < 0 || total_q < 0 || max_pages_per_seq <= 0 ||
      num_pages_total <= 0)
    return set_error(ATTN_ERR_INVALID_ARG, "bad sizes (B=%d Hq=%d Hkv=%d)", B, Hq, Hkv);
  if (Hq % Hkv != 0)
    return set_error(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (d != 64 && d != 128 && d != 256)
    return set_error(ATTN_ERR_UNSUPPORTED, "head dim %d (64, 128 or 256)", d);
  if (page_size != 16) return set_error(ATTN_ERR_UNSUPPORTED, "page size %d (16)", page_size);
  if (!(scale > 0.f) || !std::isfinite(scale))
    return set_error(ATTN_ERR_INVALID_ARG, "scale must be finite and positive");
  if (causal != 0 && causal != 1) return set_error(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (window < 0) window = 0;
  if (window > 0 && !causal)
    return set_error(ATTN_ERR_INVALID_ARG, "a sliding window requires causal");
  if (n_sink < 0 || (n_sink > 0 && window == 0))
    return set_error(ATTN_ERR_INVALID_ARG, "n_sink > 0 requires a window");
  if (static_cast<long long>(max_pages_per_seq) * page_size > (1 << 30))
    return set_error(ATTN_ERR_INVALID_ARG, "max_pages_per_seq too large");
  if (B == 0 || total_q == 0) return ATTN_OK;
  if (max_Sq == 0) return set_error(ATTN_ERR_INVALID_ARG, "max_Sq must bound the query lengths");
  if (!q || !o || !k_pages || !v_pages || !page_table || !cu_seqlens_q || !seqlens_k)
    return set_error(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(o) || !aligned16(k_pages) || !aligned16(v_pages) ||
      (reinterpret_cast<uintptr_t>(page_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) ||
      (reinterpret_cast<uintptr_t>(seqlens_k) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(sink_logit) & 3u))
    return set_error(ATTN_ERR_INVALID_ARG, "misaligned pointer");
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != ATTN_OK) return rc;
  FwdLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.o = o;
  a.lse = lse;
  a.sink = sink_logit;
  a.cu_q = cu_seqlens_q;
  a.cu_k = nullptr;
  a.page_table = page_table;
  a.seqlens_k = seqlens_k;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages_total;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = max_Sq;
  a.Skv = max_pages_per_seq * page_size;
  a.total_q = total_q;
  a.total_k = 0;
  a.d = d;
  a.scale = scale;
  a.causal = causal;
  a.window = window;
  a.n_sink = n_sink;
  a.num_sms = ds->num_sms;
  a.status = ds->status;
  a.o_sb = 0;
  a.o_ss = static_cast<long long>(Hq) * d;
  a.o_sh = d;
  if ((rc = make_map(&a.tmQ, q, d, Hq, total_q, 1, 128, "q")) != ATTN_OK) return rc;
  if ((rc = make_map(&a.tmO, o, d, Hq, total_q, 1, 128, "o")) != ATTN_OK) return rc;
  if ((rc = make_map(&a.tmK, k_pages, d, Hkv, page_size, num_pages_total, 16, "k_pages")) !=
      ATTN_OK)
    return rc;
  if ((rc = make_map(&a.tmV, v_pages, d, Hkv, page_size, num_pages_total, 16, "v_pages")) !=
      ATTN_OK)
    return rc;
  cudaError_t e = launch_attn_fwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_error(e, "attn_fwd_paged launch");
}

ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Sq) {
  if (B < 0 || Hq <= 0 || Sq < 0) return 0;
  return bwd_workspace_bytes(B, Hq, Sq);
}

}  // extern "C"

namespace {

// Every backward entry point.  sink / dsink: the logit sink per query head
// and its gradient [Hq], or both null.
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
             const int* cu_seqlens_k, int B, int Hq, int Hkv, int max_Sq, int max_Skv,
             int total_q, int total_k, int d, float scale, int causal, int window, int n_sink,
             const float* sink, float* dsink, void* workspace, size_t workspace_bytes,
             void* stream) {
  t_last_error.clear();
  if ((sink == nullptr) != (dsink == nullptr))
    return set_error(ATTN_ERR_INVALID_ARG, "sink_logit and dsink go together");
  if ((reinterpret_cast<uintptr_t>(sink) & 3u) || (reinterpret_cast<uintptr_t>(dsink) & 3u))
    return set_error(ATTN_ERR_INVALID_ARG, "misaligned sink pointer");
  const bool varlen = cu_seqlens_q != nullptr || cu_seqlens_k != nullptr;
  if (varlen && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr))
    return set_error(ATTN_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k go together");
  if (B < 0 || Hq <= 0 || Hkv <= 0 || max_Sq < 0 || max_Skv < 0)
    return set_error(ATTN_ERR_INVALID_ARG, "negative or zero size (B=%d Hq=%d Hkv=%d)", B, Hq, Hkv);
  if (varlen && (total_q < 0 || total_k < 0))
    return set_error(ATTN_ERR_INVALID_ARG, "negative total_q / total_k");
  if (Hq % Hkv != 0)
    return set_error(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (d != 64 && d != 128 && d != 256)
    return set_error(ATTN_ERR_UNSUPPORTED, "head dim %d (64, 128 or 256)", d);
  if (!(scale > 0.f) || !std::isfinite(scale))
    return set_error(ATTN_ERR_INVALID_ARG, "scale must be finite and positive");
  if (causal != 0 && causal != 1) return set_error(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (window < 0) window = 0;
  if (window > 0 && !causal)
    return set_error(ATTN_ERR_INVALID_ARG, "a sliding window requires causal");
  if (n_sink < 0 || (n_sink > 0 && window == 0))
    return set_error(ATTN_ERR_INVALID_ARG, "sink keys require a window");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B == 0 || max_Sq == 0 || (varlen && total_q == 0)) {
    // no query: dK = dV = 0 and a zero sink gradient
    const long long rows_k0 = varlen ? total_k : static_cast<long long>(B) * max_Skv;
    const size_t kv_bytes0 = static_cast<size_t>(rows_k0) * Hkv * d * 2;
    cudaError_t e = cudaSuccess;
    if (kv_bytes0 > 0) {
      if (!dk || !dv) return set_error(ATTN_ERR_INVALID_ARG, "dk and dv must be set");
      e = cudaMemsetAsync(dk, 0, kv_bytes0, st);
      if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kv_bytes0, st);
    }
    if (e == cudaSuccess && dsink) e = cudaMemsetAsync(dsink, 0, sizeof(float) * Hq, st);
    return e == cudaSuccess ? ATTN_OK : cuda_error(e, "zeroing dk/dv");
  }
  const long long rows_k = varlen ? total_k : static_cast<long long>(B) * max_Skv;
  if (!q || !o || !lse || !dout || !dq || !workspace)
    return set_error(ATTN_ERR_INVALID_ARG, "null pointer");
  if (rows_k > 0 && (!k || !v || !dk || !dv))
    return set_error(ATTN_ERR_INVALID_ARG, "k, v, dk and dv must be set");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
    return set_error(ATTN_ERR_INVALID_ARG, "tensors must be 16-byte aligned (lse 4-byte)");
  const size_t need = bwd_workspace_bytes(B, Hq, max_Sq);
  if (workspace_bytes < need)
    return set_error(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                     need);
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != ATTN_OK) return rc;
  BwdLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.sink = sink;
  a.dsink = dsink;
  a.total_q = varlen ? total_q : 0;
  a.total_k = varlen ? total_k : 0;
  const size_t rows = need / (2 * sizeof(float));
  a.ws_lse2 = static_cast<float*>(workspace);
  a.ws_d = static_cast<float*>(workspace) + rows;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sq = max_Sq;
  a.Skv = max_Skv;
  a.d = d;
  a.scale = scale;
  a.causal = causal;
  a.window = window;
  a.n_sink = n_sink;
  a.status = ds->status;
  a.num_sms = ds->num_sms;
  // Dense tensors are 4-D maps (d, H, S, B); packed ones (d, H, total, 1).
  // The d = 256 kernels stream 64-row tiles.
  const uint64_t sq = varlen ? static_cast<uint64_t>(total_q) : static_cast<uint64_t>(max_Sq);
  const uint64_t sk = varlen ? static_cast<uint64_t>(total_k) : static_cast<uint64_t>(max_Skv);
  const uint64_t nb = varlen ? 1u : static_cast<uint64_t>(B);
  const uint32_t box = d == 256 ? 64 : 128;
  if ((rc = make_map(&a.tmQ, q, d, Hq, sq, nb, box, "q")) != ATTN_OK) return rc;
  if ((rc = make_map(&a.tmDO, dout, d, Hq, sq, nb, box, "dout")) != ATTN_OK) return rc;
  if (rows_k > 0 && max_Skv > 0) {
    if ((rc = make_map(&a.tmK, k, d, Hkv, sk, nb, box, "k")) != ATTN_OK) return rc;
    if ((rc = make_map(&a.tmV, v, d, Hkv, sk, nb, box, "v")) != ATTN_OK) return rc;
  }
  cudaError_t e = launch_attn_bwd(a, st);
  return e == cudaSuccess ? ATTN_OK : cuda_error(e, "attn_bwd launch");
}

}  // namespace

extern "C" {

ATTN_API int attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                         int Hkv, int max_Sq, int max_Skv, int total_q, int total_k, int d,
                         float scale, int causal, int window, int n_sink, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv,
                  max_Sq, max_Skv, total_q, total_k, d, scale, causal, window, n_sink, nullptr,
                  nullptr, workspace, workspace_bytes, stream);
}

ATTN_API int attn_bwd_ex_sink(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                              int Hkv, int max_Sq, int max_Skv, int total_q, int total_k, int d,
                              float scale, int causal, int window, int n_sink,
                              const float* sink_logit, float* dsink, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!sink_logit || !dsink) return set_error(ATTN_ERR_INVALID_ARG, "sink_logit and dsink needed");
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv,
                  max_Sq, max_Skv, total_q, total_k, d, scale, causal, window, n_sink,
                  sink_logit, dsink, workspace, workspace_bytes, stream);
}

ATTN_API int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                      int Sq, int Skv, int d, float scale, int causal, void* workspace,
                      size_t workspace_bytes, void* stream) {
  return attn_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, nullptr, nullptr, B, Hq, Hkv, Sq, Skv, 0,
                     0, d, scale, causal, 0, 0, workspace, workspace_bytes, stream);
}

ATTN_API size_t attn_decode_workspace_size(int B, int Hq, int d, int num_splits) {
  if (B < 0 || Hq <= 0 || d <= 0 || num_splits <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * num_splits;
  // split outputs, split log-sum-exps, the request order
  return rows * d * sizeof(float) + rows * sizeof(float) + static_cast<size_t>(B) * sizeof(int);
}

}  // extern "C"

namespace {

// Every paged-decode entry point.  sink: per-head logit sink [Hq] or null.
int decode_impl(const void* q, const void* k_pages, const void* v_pages, const int* page_table,
                const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv, int d,
                int page_size, int max_pages_per_seq, int num_pages_total, int num_splits,
                float scale, const float* sink, void* workspace, size_t workspace_bytes,
                void* stream) {
  t_last_error.clear();
  if (B < 0 || Hq <= 0 || Hkv <= 0 || max_pages_per_seq <= 0 || num_pages_total <= 0)
    return set_error(ATTN_ERR_INVALID_ARG, "bad sizes");
  if (Hq % Hkv != 0)
    return set_error(ATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
  if (d != 64 && d != 128 && d != 256)
    return set_error(ATTN_ERR_UNSUPPORTED, "head dim %d (64, 128 or 256)", d);
  if (page_size != 16) return set_error(ATTN_ERR_UNSUPPORTED, "page size %d (16)", page_size);
  if (num_splits < 1 || num_splits > 64)
    return set_error(ATTN_ERR_INVALID_ARG, "num_splits %d not in [1, 64]", num_splits);
  if (!(scale > 0.f) || !std::isfinite(scale))
    return set_error(ATTN_ERR_INVALID_ARG, "scale must be finite and positive");
  if (B == 0) return ATTN_OK;
  if (!q || !k_pages || !v_pages || !page_table || !seqlens || !o || !workspace)
    return set_error(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(page_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seqlens) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(sink) & 3u))
    return set_error(ATTN_ERR_INVALID_ARG, "misaligned pointer");
  const size_t need = attn_decode_workspace_size(B, Hq, d, num_splits);
  if (workspace_bytes < need)
    return set_error(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                     need);
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != ATTN_OK) return rc;

  DecodeLaunch a;
  std::memset(&a, 0, sizeof(a));
  if ((rc = make_map(&a.tmK, k_pages, d, Hkv, page_size, num_pages_total, 16, "k_pages")) != ATTN_OK)
    return rc;
  if ((rc = make_map(&a.tmV, v_pages, d, Hkv, page_size, num_pages_total, 16, "v_pages")) != ATTN_OK)
    return rc;
  const size_t rows = static_cast<size_t>(B) * Hq * num_splits;
  a.q = q;
  a.o = o;
  a.lse = lse;
  a.sink = sink;
  a.page_table = page_table;
  a.seqlens = seqlens;
  a.ws_o = static_cast<float*>(workspace);
  a.ws_lse = static_cast<float*>(workspace) + rows * d;
  a.order = reinterpret_cast<int*>(a.ws_lse + rows);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.page = page_size;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages_total;
  a.num_splits = num_splits;
  a.scale = scale;
  a.status = ds->status;
  cudaError_t e = launch_attn_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_error(e, "attn_decode_paged launch");
}

}  // namespace

extern "C" {

ATTN_API int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                               const int* page_table, const int* seqlens, void* o, float* lse,
                               int B, int Hq, int Hkv, int d, int page_size,
                               int max_pages_per_seq, int num_pages_total, int num_splits,
                               float scale, void* workspace, size_t workspace_bytes,
                               void* stream) {
  return decode_impl(q, k_pages, v_pages, page_table, seqlens, o, lse, B, Hq, Hkv, d, page_size,
                     max_pages_per_seq, num_pages_total, num_splits, scale, nullptr, workspace,
                     workspace_bytes, stream);
}

ATTN_API int attn_decode_paged_sink(const void* q, const void* k_pages, const void* v_pages,
                                    const int* page_table, const int* seqlens, void* o,
                                    float* lse, int B, int Hq, int Hkv, int d, int page_size,
                                    int max_pages_per_seq, int num_pages_total, int num_splits,
                                    float scale, const float* sink_logit, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  return decode_impl(q, k_pages, v_pages, page_table, seqlens, o, lse, B, Hq, Hkv, d, page_size,
                     max_pages_per_seq, num_pages_total, num_splits, scale, sink_logit, workspace,
                     workspace_bytes, stream);
}

ATTN_API int attn_decode_paged_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                       const int* page_table, const int* seqlens, void* o,
                                       float* lse, int B, int Hq, int Hkv, int d, int page_size,
                                       int max_pages_per_seq, int num_pages_total, int num_splits,
                                       float scale, void* stream) {
  t_last_error.clear();
  const size_t need = attn_decode_workspace_size(B, Hq, d, num_splits);
  if (need > kNoAllocScratchBytes)
    return set_error(ATTN_ERR_INVALID_ARG,
                     "needs %zu bytes of scratch but the built-in scratch holds %zu; lower B, Hq "
                     "or num_splits, or use attn_decode_paged with a workspace",
                     need, kNoAllocScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return set_error(ATTN_ERR_UNSUPPORTED, "device %d", dev);
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_scratch_ptr[dev] == nullptr) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(scratch)");
      g_noalloc_scratch_ptr[dev] = ptr;
    }
    scratch = g_noalloc_scratch_ptr[dev];
  }
  return attn_decode_paged(q, k_pages, v_pages, page_table, seqlens, o, lse, B, Hq, Hkv, d,
                           page_size, max_pages_per_seq, num_pages_total, num_splits, scale,
                           scratch, kNoAllocScratchBytes, stream);
}

ATTN_API int attn_device_status(void* stream) {
  t_last_error.clear();
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != ATTN_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpy(&word, ds->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_error(e, "reading the status word");
  const int zero = 0;
  e = cudaMemcpy(ds->status, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_error(e, "clearing the status word");
  if (word & kStatusTimeout) return ATTN_ERR_TIMEOUT;
  if (word & kStatusBadInput) return ATTN_ERR_BAD_INPUT;
  if (word & kStatusLayout) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

ATTN_API int attn_check_wait_timeout(int limit_us, void* stream) {
  t_last_error.clear();
  if (limit_us < 1 || limit_us > 1000000)
    return set_error(ATTN_ERR_INVALID_ARG, "limit_us %d not in [1, 1000000]", limit_us);
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != ATTN_OK) return rc;
  cudaError_t e = launch_wait_timeout_check(ds->status, static_cast<uint64_t>(limit_us) * 1000u,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_error(e, "timeout check launch");
}

}  // extern "C"
