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

// ------------------------------------------------------------------ top-N
//
// Exact top-N in one CTA of 1024 threads, ties to the lower index, output ascending.
// Keys are the fp32 bit patterns mapped to an order-preserving unsigned integer; K* is
// the N-th largest key and `need` how many keys equal to K* are taken (the lowest
// indices among them).
//   A  histogram passes over the scores, 11, 11 and 10 key bits from the top, each
//      restricted to the bucket chosen so far, until the bucket holding the N-th largest
//      key has at most kTopnCap keys (one pass for most score distributions; for
//      C <= kTopnCap none: every score is a candidate)
//   B  one more pass appends that bucket's keys, with their indices, to a candidate list
//      in shared memory
//   R  in shared memory: the remaining key bits give K* and `need`; two 12-bit rounds
//      over the indices of the K*-valued candidates give idx*, the largest index taken
//   C  a last pass writes, in index order, every j with key > K* or (key == K* and
//      j <= idx*): a block-wide scan per 4096 scores
// When all 32 bits are fixed and more than kTopnCap keys still equal K*, the last pass
// instead ranks the K*-valued keys in index order with the same block-wide scans.
constexpr int kTopnThreads = 1024;
constexpr int kTopnCap = 16384;                               // candidates held in shared memory
constexpr int kTopnSmem = 2 * kTopnCap * 4 + 4096 * 4;       // keys, indices, one 4096-bin histogram

__device__ __forceinline__ unsigned int topn_scan_excl(unsigned int v, unsigned int* wsum, unsigned int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  unsigned int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[wid] = x;
  __syncthreads();
  if (wid == 0) {
    const unsigned int w = wsum[lane];
    unsigned int z = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned int y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    wsum[lane] = z - w;
    if (lane == 31) wsum[32] = z;
  }
  __syncthreads();
  const unsigned int r = wsum[wid] + x - v;
  *total = wsum[32];
  __syncthreads();
  return r;
}

// The bin holding the need-th element counted from the top bin down (desc) or from bin 0
// up (asc): out = {bin, elements still needed from it, the bin's count}.
// nbins in {1024, 2048, 4096}.
__device__ void topn_pick_bin(const unsigned int* h, int nbins, bool desc, unsigned int need, unsigned int* wsum,
                              unsigned int* out) {
  const int k = nbins / kTopnThreads;
  const int p0 = threadIdx.x * k;
  unsigned int local = 0u;
  for (int i = 0; i < k; ++i) local += h[desc ? nbins - 1 - (p0 + i) : p0 + i];
  unsigned int tot;
  unsigned int before = topn_scan_excl(local, wsum, &tot);
  if (before < need && need <= before + local) {
    for (int i = 0; i < k; ++i) {
      const int bin = desc ? nbins - 1 - (p0 + i) : p0 + i;
      const unsigned int c = h[bin];
      if (before + c >= need) {
        out[0] = static_cast<unsigned int>(bin);
        out[1] = need - before;
        out[2] = c;
        break;
      }
      before += c;
    }
  }
  __syncthreads();
}

// Sixteen consecutive scores from j0 as keys; keys past C are reported by the count n
// (all loads are issued before any key is used, so a thread keeps four in flight).
constexpr int kTopnPer = 16;
__device__ __forceinline__ void topn_load16(const float* __restrict__ s, int j0, int C, unsigned int* k, int* n) {
  if (j0 + kTopnPer <= C) {
    const float4* p = reinterpret_cast<const float4*>(s + j0);
    float4 f[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) f[u] = __ldg(p + u);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      k[4 * u] = order_key(f[u].x);
      k[4 * u + 1] = order_key(f[u].y);
      k[4 * u + 2] = order_key(f[u].z);
      k[4 * u + 3] = order_key(f[u].w);
    }
    *n = kTopnPer;
  } else {
    const int m = max(0, C - j0);
#pragma unroll
    for (int e = 0; e < kTopnPer; ++e) k[e] = e < m ? order_key(s[j0 + e]) : 0u;
    *n = m;
  }
}

__device__ __forceinline__ int topn_level_shift(int lv) { return lv == 0 ? 21 : (lv == 1 ? 10 : 0); }
__device__ __forceinline__ int topn_level_bins(int lv) { return lv == 2 ? 1024 : 2048; }

__global__ void __launch_bounds__(kTopnThreads, 1) topn_kernel(const float* __restrict__ scores, int C, int N,
                                                            int32_t* __restrict__ sel) {
  pdl_wait();  // the scores come from the kernel before
  pdl_launch_dependents();
  extern __shared__ __align__(16) unsigned int tsm[];
  unsigned int* ckey = tsm;                                 // [kTopnCap] candidate keys
  int* cidx = reinterpret_cast<int*>(tsm + kTopnCap);       // [kTopnCap] candidate indices
  unsigned int* h = tsm + 2 * kTopnCap;                     // [4096] histogram
  unsigned int* hist8 = tsm;                                // passes A: [8][2048] over the candidate list
  __shared__ unsigned int wsum[33];
  __shared__ unsigned int pick[3];
  __shared__ unsigned int s_cnt;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  unsigned int need = static_cast<unsigned int>(N);
  unsigned int prefix = 0u, fmask = 0u;  // key bits fixed so far
  int lv = 0;
  int n_c = C;
  const bool all_in_smem = C <= kTopnCap;
  if (all_in_smem) {
    for (int j = tid; j < C; j += kTopnThreads) {
      ckey[j] = order_key(scores[j]);
      cidx[j] = j;
    }
    __syncthreads();
  } else {
    // ---- A: narrow to a bucket of at most kTopnCap keys
    unsigned int bucket = 0u;
    while (true) {
      const int shift = topn_level_shift(lv), nb = topn_level_bins(lv);
      for (int i = tid; i < 8 * 2048; i += kTopnThreads) hist8[i] = 0u;
      __syncthreads();
      unsigned int* myh = hist8 + (wid & 7) * 2048;
      for (int base = 0; base < C; base += kTopnPer * kTopnThreads) {
        unsigned int k[kTopnPer];
        int n;
        topn_load16(scores, base + kTopnPer * tid, C, k, &n);
#pragma unroll
        for (int e = 0; e < kTopnPer; ++e)
          if (e < n && (k[e] & fmask) == prefix) atomicAdd(&myh[(k[e] >> shift) & (nb - 1)], 1u);
      }
      __syncthreads();
      for (int b = tid; b < nb; b += kTopnThreads) {
        unsigned int t = 0u;
#pragma unroll
        for (int c = 0; c < 8; ++c) t += hist8[c * 2048 + b];
        h[b] = t;
      }
      __syncthreads();
      topn_pick_bin(h, nb, true, need, wsum, pick);
      prefix |= pick[0] << shift;
      fmask |= static_cast<unsigned int>(nb - 1) << shift;
      need = pick[1];
      bucket = pick[2];
      ++lv;
      if (bucket <= static_cast<unsigned int>(kTopnCap) || lv == 3) break;
    }
    if (bucket > static_cast<unsigned int>(kTopnCap)) {
      // ---- every key bit is fixed and too many keys equal K*: rank them in index order
      const unsigned int kstar = prefix;
      unsigned int out = 0u, eq_seen = 0u;
      for (int base = 0; base < C; base += kTopnPer * kTopnThreads) {
        const int j0 = base + kTopnPer * tid;
        unsigned int k[kTopnPer];
        int n;
        topn_load16(scores, j0, C, k, &n);
        unsigned int n_eq = 0u;
#pragma unroll
        for (int e = 0; e < kTopnPer; ++e) n_eq += (e < n && k[e] == kstar) ? 1u : 0u;
        unsigned int eq_tot;
        unsigned int r = eq_seen + topn_scan_excl(n_eq, wsum, &eq_tot);
        unsigned int fbits = 0u;
#pragma unroll
        for (int e = 0; e < kTopnPer; ++e) {
          const bool eq = e < n && k[e] == kstar;
          if ((e < n && k[e] > kstar) || (eq && r < need)) fbits |= 1u << e;
          r += eq ? 1u : 0u;
        }
        unsigned int tot;
        unsigned int pos = out + topn_scan_excl(__popc(fbits), wsum, &tot);
#pragma unroll
        for (int e = 0; e < kTopnPer; ++e)
          if (((fbits >> e) & 1u) && pos < static_cast<unsigned int>(N)) sel[pos++] = j0 + e;
        out += tot;
        eq_seen += eq_tot;
      }
      return;
    }
    // ---- B: that bucket's keys, with their indices, into the candidate list
    if (tid == 0) s_cnt = 0u;
    __syncthreads();
    for (int base = 0; base < C; base += kTopnPer * kTopnThreads) {
      unsigned int k[kTopnPer];
      int n;
      topn_load16(scores, base + kTopnPer * tid, C, k, &n);
#pragma unroll
      for (int e = 0; e < kTopnPer; ++e) {
        const bool m = e < n && (k[e] & fmask) == prefix;
        const unsigned int bal = __ballot_sync(0xffffffffu, m);
        if (bal) {
          const int leader = __ffs(bal) - 1;
          unsigned int b0 = 0u;
          if (lane == leader) b0 = atomicAdd(&s_cnt, static_cast<unsigned int>(__popc(bal)));
          b0 = __shfl_sync(0xffffffffu, b0, leader);
          if (m) {
            const unsigned int pos = b0 + __popc(bal & ((1u << lane) - 1u));
            if (pos < static_cast<unsigned int>(kTopnCap)) {
              ckey[pos] = k[e];
              cidx[pos] = base + kTopnPer * tid + e;
            }
          }
        }
      }
    }
    __syncthreads();
    n_c = min(static_cast<int>(s_cnt), kTopnCap);
  }
  // ---- R: the remaining key bits over the candidates give K* and `need`
  for (; lv < 3; ++lv) {
    const int shift = topn_level_shift(lv), nb = topn_level_bins(lv);
    for (int i = tid; i < nb; i += kTopnThreads) h[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n_c; i += kTopnThreads) {
      const unsigned int key = ckey[i];
      if ((key & fmask) == prefix) atomicAdd(&h[(key >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    topn_pick_bin(h, nb, true, need, wsum, pick);
    prefix |= pick[0] << shift;
    fmask |= static_cast<unsigned int>(nb - 1) << shift;
    need = pick[1];
  }
  const unsigned int kstar = prefix;
  // ---- the need-th smallest index among the K*-valued candidates (C <= 2^24)
  unsigned int ip = 0u, im = 0u;
  for (int il = 0; il < 2; ++il) {
    const int shift = il == 0 ? 12 : 0;
    for (int i = tid; i < 4096; i += kTopnThreads) h[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n_c; i += kTopnThreads) {
      const unsigned int idx = static_cast<unsigned int>(cidx[i]);
      if (ckey[i] == kstar && (idx & im) == ip) atomicAdd(&h[(idx >> shift) & 4095u], 1u);
    }
    __syncthreads();
    topn_pick_bin(h, 4096, false, need, wsum, pick);
    ip |= pick[0] << shift;
    im |= 4095u << shift;
    need = pick[1];
  }
  const unsigned int idx_star = ip;
  // ---- C: every j with key > K*, or key == K* and j <= idx*, in index order
  unsigned int out = 0u;
  for (int base = 0; base < C; base += kTopnPer * kTopnThreads) {
    const int j0 = base + kTopnPer * tid;
    unsigned int k[kTopnPer];
    int n;
    if (all_in_smem) {
      n = max(0, min(kTopnPer, C - j0));
#pragma unroll
      for (int e = 0; e < kTopnPer; ++e) k[e] = e < n ? ckey[j0 + e] : 0u;
    } else {
      topn_load16(scores, j0, C, k, &n);
    }
    unsigned int fbits = 0u;
#pragma unroll
    for (int e = 0; e < kTopnPer; ++e)
      if (e < n && (k[e] > kstar || (k[e] == kstar && static_cast<unsigned int>(j0 + e) <= idx_star))) fbits |= 1u << e;
    unsigned int tot;
    unsigned int pos = out + topn_scan_excl(__popc(fbits), wsum, &tot);
#pragma unroll
    for (int e = 0; e < kTopnPer; ++e)
      if (((fbits >> e) & 1u) && pos < static_cast<unsigned int>(N)) sel[pos++] = j0 + e;
    out += tot;
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

namespace qcf {
qcf_status topn_launch(const float* scores, int C, int N, int32_t* sel, cudaStream_t st, bool pdl) {
  if (!scores || (!sel && N > 0)) return set_error(QCF_ERR_INVALID_ARG, "qcf_topn_select: NULL pointer");
  if (C < 0 || C > (1 << 24) || N < 0 || N > C) return set_error(QCF_ERR_SHAPE, "qcf_topn_select: C=%d N=%d", C, N);
  if (take_fault(4) || !aligned16(scores)) return set_error(QCF_ERR_ALIGN, "qcf_topn_select: scores not 16-byte aligned");
  if (N == 0) return QCF_OK;
  static PerDevice<cudaError_t> smem_attr;
  const cudaError_t attr = smem_attr.get(current_device(), [] {
    return cudaFuncSetAttribute(topn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTopnSmem);
  });
  if (attr != cudaSuccess) return cuda_error(attr, "qcf_topn_select: smem attribute");
  LaunchScope ls(KC_TOPN, st);
  cudaError_t e;
  if (pdl) {
    e = launch_pdl(topn_kernel, dim3(1), dim3(kTopnThreads), kTopnSmem, st, scores, C, N, sel);
  } else {
    topn_kernel<<<1, kTopnThreads, kTopnSmem, st>>>(scores, C, N, sel);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_topn_select: launch");
}
}  // namespace qcf

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
  return topn_launch(scores, C, N, sel, static_cast<cudaStream_t>(stream), false);
}

size_t qcf_topn_select_workspace_size(int C) {
  return C > kTopnCap ? topn_grid_workspace_size(C) : 0;
}

qcf_status qcf_topn_select_ws(const float* scores, int C, int N, int32_t* sel, void* ws, size_t ws_bytes,
                              void* stream) {
  if (!scores || (!sel && N > 0)) return set_error(QCF_ERR_INVALID_ARG, "qcf_topn_select_ws: NULL pointer");
  if (C < 0 || C > (1 << 24) || N < 0 || N > C)
    return set_error(QCF_ERR_SHAPE, "qcf_topn_select_ws: C=%d N=%d", C, N);
  const size_t need = qcf_topn_select_workspace_size(C);
  if (need > 0 && !ws) return set_error(QCF_ERR_INVALID_ARG, "qcf_topn_select_ws: NULL workspace");
  if (take_fault(4) || !aligned16(scores) || !aligned16(ws))
    return set_error(QCF_ERR_ALIGN, "qcf_topn_select_ws: alignment");
  if (take_fault(2) || ws_bytes < need)
    return set_error(QCF_ERR_WORKSPACE, "qcf_topn_select_ws: workspace %zu < %zu", ws_bytes, need);
  if (N == 0) return QCF_OK;
  // one CTA holds up to kTopnCap scores in shared memory; larger vectors spread over a
  // cooperative grid while all its CTAs fit on the device at once
  if (C <= kTopnCap || C > topn_grid_max_scores()) return qcf_topn_select(scores, C, N, sel, stream);
  return topn_grid_launch(scores, C, N, sel, ws, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
