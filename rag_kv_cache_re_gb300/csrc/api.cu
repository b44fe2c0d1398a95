// Library-wide plumbing: errors, device status word, fault injection, launch
// accounting, per-kernel event timing, RoPE tables and small shape helpers.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <vector>

#include "qcf_internal.cuh"

namespace qcf {

static thread_local char g_err[512] = "";
static std::atomic<int> g_fault{0};
static std::atomic<int> g_check{0};
static std::atomic<int64_t> g_launches{0};

__device__ unsigned int g_device_status = 0;

qcf_status set_error(qcf_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

qcf_status cuda_error(cudaError_t e, const char* what) {
  return set_error(QCF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool take_fault(int kind) {
  int k = kind;
  return g_fault.compare_exchange_strong(k, 0);
}

bool check_enabled() { return g_check.load() != 0; }

unsigned int* device_status_ptr() {
  static std::mutex mu;
  static std::vector<unsigned int*> per_dev;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (static_cast<int>(per_dev.size()) <= dev) per_dev.resize(dev + 1, nullptr);
  if (!per_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    per_dev[dev] = static_cast<unsigned int*>(p);
  }
  return per_dev[dev];
}

int current_device() {
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

int num_sms() {
  static std::mutex mu;
  static std::vector<int> per_dev;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  if (static_cast<int>(per_dev.size()) <= dev) per_dev.resize(dev + 1, 0);
  if (!per_dev[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    per_dev[dev] = n > 0 ? n : 1;
  }
  return per_dev[dev];
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// ------------------------------------------------------------------ timing
static const char* kClassNames[KC_COUNT] = {
    "rope_reposition", "anchor_keynorm_topk", "profile_scores", "topn_select", "gather_rows",
    "scatter_kv",      "sparse_causal_attn",  "attn_combine",   "gemm_qkv_rope", "gemm_o_resid",
    "gemm_gate_up_swiglu", "gemm_down_resid", "gemm_other",     "rmsnorm",     "embed_rows",
    "lm_head_argmax",  "misc",         "probe_gemm",     "probe_attn"};

struct TimingState {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> start, stop;
  std::vector<int> cls;
  int used = 0;
};
static TimingState& timing() {
  static TimingState t;
  return t;
}

LaunchScope::LaunchScope(KernelClass k, cudaStream_t s) : kc(k), stream(s), slot(-1) {
  count_launch();
  TimingState& t = timing();
  if (!t.on) return;
  std::lock_guard<std::mutex> lk(t.mu);
  if (t.used >= static_cast<int>(t.start.size())) {
    const int grow = 1024;
    for (int i = 0; i < grow; ++i) {
      cudaEvent_t a, b;
      if (cudaEventCreate(&a) != cudaSuccess) return;
      if (cudaEventCreate(&b) != cudaSuccess) return;
      t.start.push_back(a);
      t.stop.push_back(b);
      t.cls.push_back(0);
    }
  }
  slot = t.used++;
  t.cls[slot] = kc;
  cudaEventRecord(t.start[slot], stream);
}

LaunchScope::~LaunchScope() {
  if (slot < 0) return;
  cudaEventRecord(timing().stop[slot], stream);
}

}  // namespace qcf

using namespace qcf;

extern "C" {

const char* qcf_last_error(void) { return g_err; }

const char* qcf_version(void) { return "qcf 0.1 (sm_103a)"; }

qcf_status qcf_query_status(void* stream, uint32_t* status) {
  if (!status) return set_error(QCF_ERR_INVALID_ARG, "qcf_query_status: status is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_error(e, "qcf_query_status: stream synchronize");
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
  if (e != cudaSuccess) return cuda_error(e, "qcf_query_status: read status");
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_error(e, "qcf_query_status: clear status");
  *status = v;
  return QCF_OK;
}

qcf_status qcf_debug_set_fault(int kind) {
  if (kind < 0 || kind > 4) return set_error(QCF_ERR_INVALID_ARG, "qcf_debug_set_fault: unknown kind %d", kind);
  g_fault.store(kind);
  return QCF_OK;
}

qcf_status qcf_set_check(int on) {
  g_check.store(on ? 1 : 0);
  return QCF_OK;
}

int64_t qcf_launch_count(void) { return g_launches.load(); }

qcf_status qcf_timing_enable(int on) {
  TimingState& t = timing();
  std::lock_guard<std::mutex> lk(t.mu);
  t.on = on != 0;
  t.used = 0;
  return QCF_OK;
}

qcf_status qcf_timing_read(int max, const char** names, double* ms, int64_t* launches, int* n_classes) {
  TimingState& t = timing();
  std::lock_guard<std::mutex> lk(t.mu);
  double acc[KC_COUNT] = {0};
  int64_t cnt[KC_COUNT] = {0};
  for (int i = 0; i < t.used; ++i) {
    cudaError_t e = cudaEventSynchronize(t.stop[i]);
    if (e != cudaSuccess) return cuda_error(e, "qcf_timing_read: event synchronize");
    float f = 0.f;
    e = cudaEventElapsedTime(&f, t.start[i], t.stop[i]);
    if (e != cudaSuccess) return cuda_error(e, "qcf_timing_read: elapsed time");
    acc[t.cls[i]] += f;
    cnt[t.cls[i]] += 1;
  }
  t.used = 0;
  const int n = max < KC_COUNT ? max : KC_COUNT;
  for (int i = 0; i < n; ++i) {
    if (names) names[i] = kClassNames[i];
    if (ms) ms[i] = acc[i];
    if (launches) launches[i] = cnt[i];
  }
  if (n_classes) *n_classes = n;
  return QCF_OK;
}

qcf_status qcf_num_selected(int C, int ratio_bp, int* N) {
  if (!N) return set_error(QCF_ERR_INVALID_ARG, "qcf_num_selected: N is NULL");
  if (C < 0 || ratio_bp < 0 || ratio_bp > 10000)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_num_selected: C=%d ratio_bp=%d", C, ratio_bp);
  long long v = (static_cast<long long>(ratio_bp) * C + 9999) / 10000;
  if (v > C) v = C;
  *N = static_cast<int>(v);
  return QCF_OK;
}

qcf_status qcf_rope_table_fill_host(float* cos_host, float* sin_host, int max_pos, int D, double theta) {
  if (!cos_host || !sin_host || max_pos <= 0 || D <= 0 || (D & 1) || !(theta > 1.0))
    return set_error(QCF_ERR_INVALID_ARG, "qcf_rope_table_fill_host: bad arguments");
  const int half = D / 2;
  std::vector<double> omega(half);
  for (int k = 0; k < half; ++k) omega[k] = 1.0 / std::pow(theta, 2.0 * k / D);
  for (int p = 0; p < max_pos; ++p) {
    for (int k = 0; k < half; ++k) {
      const double a = static_cast<double>(p) * omega[k];
      cos_host[static_cast<size_t>(p) * half + k] = static_cast<float>(std::cos(a));
      sin_host[static_cast<size_t>(p) * half + k] = static_cast<float>(std::sin(a));
    }
  }
  return QCF_OK;
}

}  // extern "C"

namespace qcf {

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;  // the driver entry point is the same for every device
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                    uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle, CUtensorMapDataType dtype) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_3d(CUtensorMap* map, const void* base, const uint64_t dims[3], const uint64_t strides_bytes[2],
                    const uint32_t box[3], CUtensorMapSwizzle swizzle, CUtensorMapDataType dtype) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
  if (!fn) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
  cuuint32_t b[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, 3, const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace qcf
