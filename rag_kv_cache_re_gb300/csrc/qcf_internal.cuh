// Internal helpers shared by the qcf CUDA sources (sm_103a only).
#pragma once

#include "per_device.h"
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <utility>

#include "../../include/qcf.h"

namespace qcf {

// ------------------------------------------------------------------ host side

// Thread-local last error and status helpers (api.cu).
qcf_status set_error(qcf_status s, const char* fmt, ...);
qcf_status cuda_error(cudaError_t e, const char* what);
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Fault injection (api.cu): returns true once for the armed kind.
bool take_fault(int kind);
bool check_enabled();

// Device status word (api.cu owns the symbol).
unsigned int* device_status_ptr();

// Launch accounting and optional per-class event timing (api.cu).
enum KernelClass {
  KC_ROPE = 0, KC_ANCHOR, KC_PROFILE, KC_TOPN, KC_GATHER, KC_SCATTER, KC_ATTN, KC_ATTN_COMBINE,
  KC_GEMM_QKV, KC_GEMM_O, KC_GEMM_GU, KC_GEMM_DOWN, KC_GEMM_OTHER, KC_RMSNORM, KC_EMBED,
  KC_LMHEAD, KC_MISC, KC_GEMM_PROBE, KC_ATTN_PROBE, KC_COUNT
};
struct LaunchScope {
  LaunchScope(KernelClass kc, cudaStream_t s);
  ~LaunchScope();
  KernelClass kc;
  cudaStream_t stream;
  int slot;
};
void count_launch();

// TMA descriptor encoding through the driver entry point (gemm.cu / attention.cu).
bool encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swizzle, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);

// Rank-3 tiled map: dims innermost first, strides of dims 1 and 2 in bytes.
bool encode_tmap_3d(CUtensorMap* map, const void* base, const uint64_t dims[3], const uint64_t strides_bytes[2],
                    const uint32_t box[3], CUtensorMapSwizzle swizzle,
                    CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Device SM count (cached per device).
int num_sms();

// The current device, or -1 when it cannot be read (per-device set-up keys on it).
int current_device();

// Programmatic dependent launch.  A kernel launched this way may start while its
// predecessor in the stream drains (set-up of barriers, tensor memory and constant
// operands overlaps the predecessor's tail); it must execute pdl_wait() before it
// touches anything the predecessor (or earlier work) produced.  Only kernels that do
// so are launched with it.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Internal launchers (no argument checks; callers validated).
cudaError_t launch_rmsnorm(const float* x, int n, int d, const __nv_bfloat16* g, float eps,
                           __nv_bfloat16* h, cudaStream_t st, bool pdl = false);

// GEMM epilogue parameters (gemm.cu).
enum EpiKind { EPI_STORE_BF16 = 0, EPI_ADD_F32 = 1, EPI_QKV_ROPE = 2, EPI_SWIGLU = 3 };
struct EpiParams {
  void* out;               // STORE_BF16: bf16 [M][ldo]; ADD_F32: fp32 [M][ldo]; SWIGLU: bf16 [M][ldo]
  int ldo;
  // QKV_ROPE
  __nv_bfloat16* q_out;    // [M][Hq*D]
  __nv_bfloat16* k_cache;  // [T][Hkv*D]
  __nv_bfloat16* v_cache;
  const int32_t* rope_pos;
  const int32_t* cache_row;
  const float* cos_t;
  const float* sin_t;
  int Hq, Hkv, D, T, max_pos;
  unsigned int* status;    // device status word for index-check failures
};
// GEMM workspace: tile arrival counters (reset to zero by every completed launch)
// followed by fp32 partial slots.  gemm_ws_prepare zeroes the counters once, after
// which launches given ws_zeroed skip their own counter reset.
size_t gemm_workspace_size(int M, int N, int K);
qcf_status gemm_ws_prepare(void* ws, size_t ws_bytes, cudaStream_t st);
qcf_status gemm_launch(EpiKind epi, const __nv_bfloat16* A, int M, int K, const __nv_bfloat16* W, int N,
                       const EpiParams& ep, void* ws, size_t ws_bytes, cudaStream_t st, KernelClass kc,
                       bool w_kn = false, bool pdl = false, bool ws_zeroed = false);

// Row kernels (rows.cu).
cudaError_t launch_embed(const __nv_bfloat16* embed, int vocab, int d, const int32_t* ids, const int32_t* rows,
                         int row_offset, int n, float* x, cudaStream_t st, bool pdl = false);
// best_ws: qcf_lm_head_workspace_size() bytes (one argmax key per CTA)
cudaError_t launch_lm_head(const qcf_model* m, const float* x_last, float* logits, int32_t* token, void* best_ws,
                           cudaStream_t st, bool pdl = false);
cudaError_t launch_reposition(const __nv_bfloat16* src, __nv_bfloat16* dst, int64_t n_rows, int Hkv, int D,
                              const int32_t* seg_start, const int32_t* seg_delta, int n_seg, const qcf_rope_table* t,
                              cudaStream_t st);

cudaError_t launch_stage_scatter(const __nv_bfloat16* stK, const __nv_bfloat16* stV, const int32_t* src_row,
                                 const int32_t* delta, int64_t n_rows, int64_t staged_rows, int Hkv, int D,
                                 const qcf_rope_table* t, __nv_bfloat16* K, __nv_bfloat16* V, bool do_k, bool do_v,
                                 cudaStream_t st);

// KV deviation of fresh rows against the cache (select.cu).
cudaError_t launch_kv_deviation(const __nv_bfloat16* k_new, const __nv_bfloat16* v_new, const int32_t* pos, int n,
                                const __nv_bfloat16* K, const __nv_bfloat16* V, int T, int width, float* dev,
                                cudaStream_t st);

// Critical-layer profiling on tcgen05 for head dim 128 (profile_tc.cu).
size_t profile_tc_workspace_size(int nq, int C, int Hq, int Hkv);
qcf_status profile_tc_launch(const __nv_bfloat16* q, const __nv_bfloat16* K, int nq, int C, int Hq, int Hkv,
                             float scale, float* scores, void* ws, cudaStream_t st);
constexpr int kProfileTcMaxGroup = 16;  // heads per KV head served by the tensor-core profile
// top-N on one CTA (select.cu): the body of qcf_topn_select, optionally launched
// programmatically (the kernel waits for its predecessor before reading the scores)
qcf_status topn_launch(const float* scores, int C, int N, int32_t* sel, cudaStream_t st, bool pdl);
// exact top-N over a cooperative grid (topn_grid.cu); workspace and launch
size_t topn_grid_workspace_size(int C);
int topn_grid_max_scores();  // largest C whose CTAs all stay resident on the current device (0 if unknown)
qcf_status topn_grid_launch(const float* scores, int C, int N, int32_t* sel, void* ws, cudaStream_t st);

// Attention internals (attention.cu).
size_t attn_workspace_size(int n, int T, int Hq, int Hkv, int D);
qcf_status attn_launch(const __nv_bfloat16* q, const int32_t* pos, int n, const __nv_bfloat16* K,
                       const __nv_bfloat16* V, int T, int Hq, int Hkv, int D, float scale, __nv_bfloat16* o,
                       float* lse, void* ws, size_t ws_bytes, cudaStream_t st, KernelClass kc = KC_ATTN,
                       bool pdl = false, const int32_t* key0 = nullptr);   // key0: per row block key base (D = 128)

}  // namespace qcf

// Device-side wrappers of the PTX instructions the kernels use (mbarrier, TMA, tcgen05).
#include "ptx.cuh"
