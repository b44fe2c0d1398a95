// Selection kernels: key-norm anchors per chunk and exact top-N by radix select.
#include "qcf_internal.cuh"

namespace qcf {

constexpr int kMaxChunks = 512;
constexpr int kMaxChunkLen = 16384;
constexpr int kMaxAnchor = 64;

struct ChunkTable {
  int n_chunks;
  int start[kMaxChunks + 1];
};

// Larger key <=> larger value; -0.0 maps to the key of +0.0.
__device__ __forceinline__ unsigned int order_key(float f) {
  unsigned int b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) == 0u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// One CTA per chunk: squared key norms over all H_kv*D entries (fp32, fixed
// reduction order), then n_anchor rounds of block argmax (largest norm, lowest
// index on ties), written ascending.
__global__ void __launch_bounds__(256) anchor_keynorm_kernel(const __nv_bfloat16* __restrict__ K, int HD,
                                                             const ChunkTable ct, int n_anchor,
                                                             int32_t* __restrict__ anchor_idx,
                                                             float* __restrict__ norms) {
  extern __shared__ float nrm[];
  __shared__ float bv[8];
  __shared__ int bi[8];
  __shared__ int chosen[kMaxAnchor];
  const int c = blockIdx.x;
  const int s0 = ct.start[c], len = ct.start[c + 1] - s0;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int i = wid; i < len; i += 8) {
    const uint4* row = reinterpret_cast<const uint4*>(K + static_cast<int64_t>(s0 + i) * HD);
    float ss = 0.f;
    for (int j = lane; j < HD / 8; j += 32) {
      const uint4 u = row[j];
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 f = __bfloat1622float2(h[t]);
        ss = fmaf(f.x, f.x, ss);
        ss = fmaf(f.y, f.y, ss);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) {
      nrm[i] = ss;
      if (norms) norms[s0 + i] = sqrtf(ss);
    }
  }
  __syncthreads();
  for (int a = 0; a < n_anchor; ++a) {
    float best = -1.f;
    int bidx = 0x7FFFFFFF;
    for (int i = threadIdx.x; i < len; i += blockDim.x) {
      const float v = nrm[i];
      if (v > best) {   // strided ascending scan: the first of equal values is the lowest index
        best = v;
        bidx = i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
      if (ov > best || (ov == best && oi < bidx)) {
        best = ov;
        bidx = oi;
      }
    }
    if (lane == 0) {
      bv[wid] = best;
      bi[wid] = bidx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float b = bv[0];
      int ix = bi[0];
      for (int w = 1; w < 8; ++w)
        if (bv[w] > b || (bv[w] == b && bi[w] < ix)) {
          b = bv[w];
          ix = bi[w];
        }
      chosen[a] = ix;
      nrm[ix] = -2.f;   // below every squared norm
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    for (int i = 1; i < n_anchor; ++i) {   // insertion sort, ascending
      const int v = chosen[i];
      int j = i - 1;
      while (j >= 0 && chosen[j] > v) {
        chosen[j + 1] = chosen[j];
        --j;
      }
      chosen[j + 1] = v;
    }
    for (int i = 0; i < n_anchor; ++i) anchor_idx[c * n_anchor + i] = chosen[i];
  }
}

// Exact top-N in one CTA of 1024 threads.
// (1) Radix select, 8 bits at a time from the top, finds the key K* of the N-th
//     largest value and `need`, how many elements equal to K* are taken.
// (2) Compaction in index order: an element is selected if key > K*, or if key == K*
//     and fewer than `need` equal keys precede it.  Output is ascending.
constexpr int kTopnThreads = 1024;
__global__ void __launch_bounds__(kTopnThreads) topn_kernel(const float* __restrict__ scores, int C, int N,
                                                            int32_t* __restrict__ sel) {
  __shared__ unsigned int hist[32][256];
  __shared__ unsigned int tot[256];
  __shared__ unsigned int s_prefix, s_need;
  __shared__ unsigned int wsum_a[32], wsum_b[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  unsigned int prefix = 0u, mask = 0u, need = static_cast<unsigned int>(N);
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 32 * 256; i += kTopnThreads) (&hist[0][0])[i] = 0u;
    __syncthreads();
    for (int base = 0; base < C; base += kTopnThreads) {
      const int j = base + threadIdx.x;
      const bool valid = j < C;
      const unsigned int k = valid ? order_key(scores[j]) : 0u;
      const bool part = valid && ((k & mask) == prefix);
      const unsigned int digit = (k >> shift) & 255u;
      // warp-aggregated increment: one atomic per distinct digit in the warp
      const unsigned int peers = __match_any_sync(0xffffffffu, part ? digit : 0x100u);
      if (part && (__ffs(peers) - 1) == lane) atomicAdd(&hist[wid][digit], __popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 256) {
      unsigned int t = 0u;
      for (int w = 0; w < 32; ++w) t += hist[w][threadIdx.x];
      tot[threadIdx.x] = t;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned int cum = 0u;
      int d = 255;
      for (; d > 0; --d) {
        if (cum + tot[d] >= need) break;
        cum += tot[d];
      }
      s_prefix = prefix | (static_cast<unsigned int>(d) << shift);
      s_need = need - cum;
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix == K*, need = number of K*-valued elements to take (lowest indices first)
  unsigned int eq_seen = 0u, out_seen = 0u;
  for (int base = 0; base < C; base += kTopnThreads) {
    const int j = base + threadIdx.x;
    const bool valid = j < C;
    const unsigned int k = valid ? order_key(scores[j]) : 0u;
    const bool gt = valid && k > prefix;
    const bool eq = valid && k == prefix;
    const unsigned int eq_b = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) wsum_a[wid] = __popc(eq_b);
    __syncthreads();
    if (wid == 0) {   // exclusive scan of per-warp equal counts
      const unsigned int v = wsum_a[lane];
      unsigned int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      wsum_a[lane] = x - v;
      if (lane == 31) wsum_b[0] = x;   // tile total of equals (temporarily)
    }
    __syncthreads();
    const unsigned int eq_rank = eq_seen + wsum_a[wid] + __popc(eq_b & ((1u << lane) - 1u));
    const unsigned int eq_tile = wsum_b[0];
    const bool take = gt || (eq && eq_rank < need);
    const unsigned int tk_b = __ballot_sync(0xffffffffu, take);
    __syncthreads();
    if (lane == 0) wsum_a[wid] = __popc(tk_b);
    __syncthreads();
    if (wid == 0) {
      const unsigned int v = wsum_a[lane];
      unsigned int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      wsum_a[lane] = x - v;
      if (lane == 31) wsum_b[1] = x;
    }
    __syncthreads();
    if (take) sel[out_seen + wsum_a[wid] + __popc(tk_b & ((1u << lane) - 1u))] = j;
    eq_seen += eq_tile;
    out_seen += wsum_b[1];
    __syncthreads();
  }
}

// ------------------------------------------------------------------ KV deviation (CacheBlend HKVD)

__device__ __forceinline__ float sqdiff8(const uint4 a, const uint4 b) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 u = __bfloat1622float2(x[i]), v = __bfloat1622float2(y[i]);
    const float d0 = u.x - v.x, d1 = u.y - v.y;
    acc = fmaf(d0, d0, fmaf(d1, d1, acc));
  }
  return acc;
}

// dev[i] = |k_new[i] - K[pos[i]]|^2 + |v_new[i] - V[pos[i]]|^2 over the row's width
// entries; one warp per row, 16-byte loads.
__global__ void kv_deviation_kernel(const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
                                    const int32_t* __restrict__ pos, int n, const __nv_bfloat16* __restrict__ K,
                                    const __nv_bfloat16* __restrict__ V, int T, int width, float* __restrict__ dev,
                                    unsigned int* status) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n) return;
  const int p = pos[warp];
  if (p < 0 || p >= T) {
    if (lane == 0) {
      flag_status(status, QCF_DEV_BAD_INDEX);
      dev[warp] = 0.f;
    }
    return;
  }
  const uint4* a = reinterpret_cast<const uint4*>(k_new + static_cast<int64_t>(warp) * width);
  const uint4* b = reinterpret_cast<const uint4*>(K + static_cast<int64_t>(p) * width);
  const uint4* c = reinterpret_cast<const uint4*>(v_new + static_cast<int64_t>(warp) * width);
  const uint4* d = reinterpret_cast<const uint4*>(V + static_cast<int64_t>(p) * width);
  float acc = 0.f;
  for (int i = lane; i < width / 8; i += 32) acc += sqdiff8(a[i], b[i]) + sqdiff8(c[i], d[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) dev[warp] = acc;
}

cudaError_t launch_kv_deviation(const __nv_bfloat16* k_new, const __nv_bfloat16* v_new, const int32_t* pos, int n,
                                const __nv_bfloat16* K, const __nv_bfloat16* V, int T, int width, float* dev,
                                cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  LaunchScope ls(KC_MISC, st);
  kv_deviation_kernel<<<(n + 7) / 8, 256, 0, st>>>(k_new, v_new, pos, n, K, V, T, width, dev, device_status_ptr());
  return cudaGetLastError();
}

}  // namespace qcf

using namespace qcf;

extern "C" {

qcf_status qcf_anchor_keynorm_topk(const qcf_bf16* K, const int32_t* chunk_start, int n_chunks, int Hkv, int D,
                                   int n_anchor, int32_t* anchor_idx, float* norms, void* stream) {
  if (!K || !chunk_start || !anchor_idx) return set_error(QCF_ERR_INVALID_ARG, "qcf_anchor_keynorm_topk: NULL pointer");
  if (n_chunks <= 0 || n_chunks > kMaxChunks || Hkv <= 0 || (D != 16 && D != 64 && D != 128) || n_anchor < 0 ||
      n_anchor > kMaxAnchor)
    return set_error(QCF_ERR_SHAPE, "qcf_anchor_keynorm_topk: n_chunks=%d Hkv=%d D=%d n_anchor=%d", n_chunks, Hkv, D,
                     n_anchor);
  if (take_fault(4) || !aligned16(K)) return set_error(QCF_ERR_ALIGN, "qcf_anchor_keynorm_topk: K not 16-byte aligned");
  ChunkTable ct;
  ct.n_chunks = n_chunks;
  int max_len = 0;
  if (chunk_start[0] != 0) return set_error(QCF_ERR_SHAPE, "qcf_anchor_keynorm_topk: chunk_start[0] must be 0");
  for (int c = 0; c <= n_chunks; ++c) {
    ct.start[c] = chunk_start[c];
    if (c > 0) {
      const int len = chunk_start[c] - chunk_start[c - 1];
      if (len < n_anchor || len > kMaxChunkLen)
        return set_error(QCF_ERR_SHAPE, "qcf_anchor_keynorm_topk: chunk %d length %d (need %d..%d)", c - 1, len,
                         n_anchor, kMaxChunkLen);
      max_len = len > max_len ? len : max_len;
    }
  }
  if (n_anchor == 0) return QCF_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t smem = static_cast<size_t>(max_len) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(anchor_keynorm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_error(e, "qcf_anchor_keynorm_topk: smem attribute");
  }
  LaunchScope ls(KC_ANCHOR, st);
  anchor_keynorm_kernel<<<n_chunks, 256, smem, st>>>(reinterpret_cast<const __nv_bfloat16*>(K), Hkv * D, ct, n_anchor,
                                                     anchor_idx, norms);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_anchor_keynorm_topk: launch");
}

qcf_status qcf_kv_deviation(const qcf_bf16* k_new, const qcf_bf16* v_new, const int32_t* pos, int n,
                            const qcf_bf16* K_cache, const qcf_bf16* V_cache, int T, int Hkv, int D, float* dev,
                            void* stream) {
  if (!k_new || !v_new || !pos || !K_cache || !V_cache || !dev)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_kv_deviation: NULL pointer");
  if (n < 0 || T < 0 || Hkv <= 0 || D <= 0 || (Hkv * D) % 8)
    return set_error(QCF_ERR_SHAPE, "qcf_kv_deviation: n=%d T=%d Hkv=%d D=%d", n, T, Hkv, D);
  if (take_fault(4) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(K_cache) || !aligned16(V_cache))
    return set_error(QCF_ERR_ALIGN, "qcf_kv_deviation: alignment");
  cudaError_t e = launch_kv_deviation(reinterpret_cast<const __nv_bfloat16*>(k_new),
                                      reinterpret_cast<const __nv_bfloat16*>(v_new), pos, n,
                                      reinterpret_cast<const __nv_bfloat16*>(K_cache),
                                      reinterpret_cast<const __nv_bfloat16*>(V_cache), T, Hkv * D, dev,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_kv_deviation: launch");
}

qcf_status qcf_topn_select(const float* scores, int C, int N, int32_t* sel, void* stream) {
  if (!scores || (!sel && N > 0)) return set_error(QCF_ERR_INVALID_ARG, "qcf_topn_select: NULL pointer");
  if (C < 0 || C > (1 << 24) || N < 0 || N > C) return set_error(QCF_ERR_SHAPE, "qcf_topn_select: C=%d N=%d", C, N);
  if (take_fault(4) || !aligned16(scores)) return set_error(QCF_ERR_ALIGN, "qcf_topn_select: scores not 16-byte aligned");
  if (N == 0) return QCF_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LaunchScope ls(KC_TOPN, st);
  topn_kernel<<<1, kTopnThreads, 0, st>>>(scores, C, N, sel);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_topn_select: launch");
}

}  // extern "C"
