// Calibration of the special-function unit's exp2 rate (the ceiling of the critical-layer
// profile, which evaluates two exponentials per score-row element).
#include "qcf_internal.cuh"

namespace qcf {

// Eight independent chains of ex2.approx per thread: every exponential depends only on
// its own chain, so the rate is the unit's issue rate, not its latency.
__global__ void __launch_bounds__(256) ex2_rate_kernel(float* out, int iters) {
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = -0.0625f * static_cast<float>(j + 1) - 1e-7f * static_cast<float>(threadIdx.x);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = -fast_exp2(a[j]);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += a[j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace qcf

using namespace qcf;

extern "C" {

qcf_status qcf_calibrate_exp2_rate(float* scratch, size_t scratch_bytes, double* per_second, void* stream) {
  if (!scratch || !per_second) return set_error(QCF_ERR_INVALID_ARG, "qcf_calibrate_exp2_rate: NULL pointer");
  const int blocks = num_sms() * 8, threads = 256, iters = 4096;
  if (scratch_bytes < static_cast<size_t>(blocks) * threads * sizeof(float))
    return set_error(QCF_ERR_WORKSPACE, "qcf_calibrate_exp2_rate: scratch %zu < %zu bytes", scratch_bytes,
                     static_cast<size_t>(blocks) * threads * sizeof(float));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t a = nullptr, b = nullptr;
  cudaError_t e = cudaEventCreate(&a);
  if (e == cudaSuccess) e = cudaEventCreate(&b);
  float best = 0.f;
  for (int rep = 0; rep < 3 && e == cudaSuccess; ++rep) {
    if ((e = cudaEventRecord(a, st)) != cudaSuccess) break;
    ex2_rate_kernel<<<blocks, threads, 0, st>>>(scratch, iters);
    if ((e = cudaGetLastError()) != cudaSuccess || (e = cudaEventRecord(b, st)) != cudaSuccess ||
        (e = cudaEventSynchronize(b)) != cudaSuccess)
      break;
    float ms = 0.f;
    if ((e = cudaEventElapsedTime(&ms, a, b)) != cudaSuccess) break;
    if (rep > 0 && (best == 0.f || ms < best)) best = ms;
  }
  if (a) cudaEventDestroy(a);
  if (b) cudaEventDestroy(b);
  if (e != cudaSuccess) return cuda_error(e, "qcf_calibrate_exp2_rate");
  *per_second = 8.0 * iters * static_cast<double>(blocks) * threads / (static_cast<double>(best) * 1e-3);
  return QCF_OK;
}

}  // extern "C"
