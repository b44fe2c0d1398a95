// Row-wise HBM-bound kernels: RoPE re-rotation of reused keys, row gather and
// K/V scatter, embedding rows, RMSNorm, and the LM head with argmax.
#include <algorithm>
#include <cstring>

#include "qcf_internal.cuh"

namespace qcf {

constexpr int kMaxSeg = 512;
struct SegTable {
  int n_seg;
  int start[kMaxSeg + 1];
  int delta[kMaxSeg];
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float* f) {
  uint4 u;
  u.x = pack_bf16x2(f[0], f[1]);
  u.y = pack_bf16x2(f[2], f[3]);
  u.z = pack_bf16x2(f[4], f[5]);
  u.w = pack_bf16x2(f[6], f[7]);
  return u;
}

// Pairs (a_i, b_i) = (x_k, x_{k+D/2}) turned by angles with cosines c and sines s.
// Every product and sum is rounded on its own (no contraction into FMAs), so all
// kernels that re-rotate keys give the same bits for the same inputs.
__device__ __forceinline__ void rotate8(const float* a, const float* b, const float* c, const float* s, float* o1,
                                        float* o2) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    o1[i] = __fsub_rn(__fmul_rn(a[i], c[i]), __fmul_rn(b[i], s[i]));
    o2[i] = __fadd_rn(__fmul_rn(b[i], c[i]), __fmul_rn(a[i], s[i]));
  }
}

__device__ __forceinline__ void load_angles8(const float* cos_t, const float* sin_t, int delta, int half, int k0,
                                             float* c, float* s) {
  const float4* cp = reinterpret_cast<const float4*>(cos_t + static_cast<size_t>(delta) * half + k0);
  const float4* sp = reinterpret_cast<const float4*>(sin_t + static_cast<size_t>(delta) * half + k0);
  *reinterpret_cast<float4*>(c) = cp[0];
  *reinterpret_cast<float4*>(c + 4) = cp[1];
  *reinterpret_cast<float4*>(s) = sp[0];
  *reinterpret_cast<float4*>(s + 4) = sp[1];
}

// One thread per (row, kv head, group of 8 pair indices k..k+7): the pairs
// (k, k + D/2) of the row's segment turn by delta * omega_k from the fp32 table.
__global__ void __launch_bounds__(256) rope_reposition_kernel(const __nv_bfloat16* __restrict__ src,
                                                              __nv_bfloat16* __restrict__ dst, int64_t n_rows,
                                                              int Hkv, int D, const float* __restrict__ cos_t,
                                                              const float* __restrict__ sin_t,
                                                              const SegTable seg) {
  const int half = D / 2;
  const int groups = half / 8;
  const int64_t per_row = static_cast<int64_t>(Hkv) * groups;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tid >= n_rows * per_row) return;
  const int64_t row = tid / per_row;
  const int rem = static_cast<int>(tid - row * per_row);
  const int h = rem / groups;
  const int k0 = (rem - h * groups) * 8;
  // segment containing `row`: largest s with start[s] <= row
  int lo = 0, hi = seg.n_seg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seg.start[mid] <= row) lo = mid; else hi = mid - 1;
  }
  const int delta = seg.delta[lo];
  const size_t base = static_cast<size_t>(row) * Hkv * D + static_cast<size_t>(h) * D;
  float a[8], b[8], c[8], s[8];
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + base + k0), a);
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(src + base + half + k0), b);
  load_angles8(cos_t, sin_t, delta, half, k0, c, s);
  float o1[8], o2[8];
  rotate8(a, b, c, s, o1, o2);
  *reinterpret_cast<uint4*>(dst + base + k0) = f32_to_bf16x8(o1);
  *reinterpret_cast<uint4*>(dst + base + half + k0) = f32_to_bf16x8(o2);
}

// Batched requests share a staging copy of each distinct chunk's layer K/V; this
// writes one request's cache rows from it: row i takes staging row src_row[i], its K
// turned by R(delta[i]) (the request's offset of that chunk) when do_k, its V copied
// when do_v.  One thread per (row, kv head, group of 8 pair indices).
__global__ void __launch_bounds__(256) stage_scatter_kernel(const __nv_bfloat16* __restrict__ stK,
                                                            const __nv_bfloat16* __restrict__ stV,
                                                            const int32_t* __restrict__ src_row,
                                                            const int32_t* __restrict__ delta, int64_t n_rows,
                                                            int64_t staged_rows, int Hkv, int D,
                                                            const float* __restrict__ cos_t,
                                                            const float* __restrict__ sin_t, int max_pos,
                                                            __nv_bfloat16* __restrict__ K, __nv_bfloat16* __restrict__ V,
                                                            int do_k, int do_v, unsigned int* status) {
  const int half = D / 2;
  const int groups = half / 8;
  const int64_t per_row = static_cast<int64_t>(Hkv) * groups;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tid >= n_rows * per_row) return;
  const int64_t row = tid / per_row;
  const int rem = static_cast<int>(tid - row * per_row);
  const int h = rem / groups;
  const int k0 = (rem - h * groups) * 8;
  const int64_t sr = src_row[row];
  const int dl = delta[row];
  if (sr < 0 || sr >= staged_rows || dl < 0 || dl >= max_pos) {
    if (k0 == 0 && h == 0) flag_status(status, QCF_DEV_BAD_INDEX);
    return;
  }
  const size_t sb = static_cast<size_t>(sr) * Hkv * D + static_cast<size_t>(h) * D;
  const size_t db = static_cast<size_t>(row) * Hkv * D + static_cast<size_t>(h) * D;
  if (do_k) {
    float a[8], b[8], c[8], s[8], o1[8], o2[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(stK + sb + k0), a);
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(stK + sb + half + k0), b);
    load_angles8(cos_t, sin_t, dl, half, k0, c, s);
    rotate8(a, b, c, s, o1, o2);
    *reinterpret_cast<uint4*>(K + db + k0) = f32_to_bf16x8(o1);
    *reinterpret_cast<uint4*>(K + db + half + k0) = f32_to_bf16x8(o2);
  }
  if (do_v) {
    *reinterpret_cast<uint4*>(V + db + k0) = *reinterpret_cast<const uint4*>(stV + sb + k0);
    *reinterpret_cast<uint4*>(V + db + half + k0) = *reinterpret_cast<const uint4*>(stV + sb + half + k0);
  }
}

// dst[i] = src[idx[i]] (rows of `width` bf16, width % 8 == 0); one warp per row.
__global__ void gather_rows_kernel(const __nv_bfloat16* __restrict__ src, int64_t src_rows, int width,
                                   const int32_t* __restrict__ idx, int n, __nv_bfloat16* __restrict__ dst,
                                   unsigned int* status, int check) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n) return;
  const int64_t r = idx[warp];
  if (r < 0 || r >= src_rows) {
    if (lane == 0) flag_status(status, QCF_DEV_BAD_INDEX);
    return;
  }
  (void)check;
  const uint4* s = reinterpret_cast<const uint4*>(src + r * width);
  uint4* d = reinterpret_cast<uint4*>(dst + static_cast<int64_t>(warp) * width);
  for (int i = lane; i < width / 8; i += 32) d[i] = s[i];
}

// K_cache[pos[i]] = k_new[i], V_cache[pos[i]] = v_new[i]; one warp per row.
__global__ void scatter_kv_kernel(const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
                                  const int32_t* __restrict__ pos, int n, int width, __nv_bfloat16* __restrict__ Kc,
                                  __nv_bfloat16* __restrict__ Vc, int T, unsigned int* status) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n) return;
  const int p = pos[warp];
  if (p < 0 || p >= T) {
    if (lane == 0) flag_status(status, QCF_DEV_BAD_INDEX);
    return;
  }
  const uint4* ks = reinterpret_cast<const uint4*>(k_new + static_cast<int64_t>(warp) * width);
  const uint4* vs = reinterpret_cast<const uint4*>(v_new + static_cast<int64_t>(warp) * width);
  uint4* kd = reinterpret_cast<uint4*>(Kc + static_cast<int64_t>(p) * width);
  uint4* vd = reinterpret_cast<uint4*>(Vc + static_cast<int64_t>(p) * width);
  for (int i = lane; i < width / 8; i += 32) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

// x[i] = float(embed[ids[rows[i]]]); rows may be NULL (identity). One warp per row.
__global__ void embed_rows_kernel(const __nv_bfloat16* __restrict__ embed, int vocab, int d,
                                  const int32_t* __restrict__ ids, const int32_t* __restrict__ rows, int row_offset,
                                  int n, float* __restrict__ x, unsigned int* status) {
  pdl_wait();  // ids and the row table may come from the kernel before
  pdl_launch_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n) return;
  const int r = rows ? rows[warp] : row_offset + warp;
  const int tok = ids[r];
  if (tok < 0 || tok >= vocab) {
    if (lane == 0) flag_status(status, QCF_DEV_BAD_INDEX);
    return;
  }
  const uint4* s = reinterpret_cast<const uint4*>(embed + static_cast<int64_t>(tok) * d);
  float4* o = reinterpret_cast<float4*>(x + static_cast<int64_t>(warp) * d);
  for (int i = lane; i < d / 8; i += 32) {
    float f[8];
    bf16x8_to_f32(s[i], f);
    o[2 * i] = make_float4(f[0], f[1], f[2], f[3]);
    o[2 * i + 1] = make_float4(f[4], f[5], f[6], f[7]);
  }
}

// h = x / sqrt(mean(x^2) + eps) * g with fp32 statistics.  One CTA of 256 threads
// per row: the row (d <= 8192) is read once into registers, 4 float4 per thread,
// so every load of the row is in flight at once.
constexpr int kNormThreads = 256;
constexpr int kNormVec = 8;   // float4 per thread: d <= 256 * 4 * 8 = 8192
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const float* __restrict__ x, int n, int d,
                                                               const __nv_bfloat16* __restrict__ g, float eps,
                                                               __nv_bfloat16* __restrict__ h) {
  __shared__ float red[kNormThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<int64_t>(row) * d);
  const int nv = d / 4;
  float4 v[kNormVec];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) {
    const int i = threadIdx.x + k * kNormThreads;
    v[k] = i < nv ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[wid] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float inv = rsqrtf(tot / static_cast<float>(d) + eps);
  uint2* hr = reinterpret_cast<uint2*>(h + static_cast<int64_t>(row) * d);
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(g);
#pragma unroll
  for (int k = 0; k < kNormVec; ++k) {
    const int i = threadIdx.x + k * kNormThreads;
    if (i < nv) {
      const float2 ga = __bfloat1622float2(g2[2 * i]);
      const float2 gb = __bfloat1622float2(g2[2 * i + 1]);
      uint2 o;
      o.x = pack_bf16x2(v[k].x * inv * ga.x, v[k].y * inv * ga.y);
      o.y = pack_bf16x2(v[k].z * inv * gb.x, v[k].w * inv * gb.y);
      hr[i] = o;
    }
  }
}

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  const unsigned int b = __float_as_uint(v);
  const unsigned int ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(ord) << 32) | static_cast<unsigned int>(0xFFFFFFFFu - idx);
}

// logits = W_lm * RMSNorm(x_last) * g (fp32 h kept in shared memory); argmax as the
// largest (orderable value, inverted index) key, so ties keep the lowest index: each
// CTA writes its best key to its own slot (nothing to clear first), and
// argmax_finalize_kernel takes the largest slot.  One warp per vocabulary row, eight
// 16-byte weight loads per lane in flight: the first batch of a warp's first row is
// requested before the dependency wait (the weights are constant), the next row's
// while the current one is reduced.
constexpr int kLmLoads = 8;
__global__ void __launch_bounds__(256, 4) lm_head_kernel(const float* __restrict__ x_last, int d, int vocab,
                                                         const __nv_bfloat16* __restrict__ g, float eps,
                                                         const __nv_bfloat16* __restrict__ W,
                                                         float* __restrict__ logits,
                                                         unsigned long long* __restrict__ best) {
  extern __shared__ float hs[];
  __shared__ float red[8];
  __shared__ unsigned long long bred[8];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int n8 = d / 8;                    // 16-byte pieces of a row
  const int iters = (n8 + 32 * kLmLoads - 1) / (32 * kLmLoads);
  uint4 wv[kLmLoads];
  auto issue = [&](int row, int it) {      // pieces lane + 32 (it * kLmLoads + u) of `row`
    const uint4* wr = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(row) * d);
#pragma unroll
    for (int u = 0; u < kLmLoads; ++u) {
      const int i = lane + 32 * (it * kLmLoads + u);
      if (i < n8) wv[u] = __ldcs(wr + i);
    }
  };
  const int nwarps = gridDim.x * 8;
  int v = blockIdx.x * 8 + wid;
  if (v < vocab) issue(v, 0);
  pdl_wait();  // x_last comes from the kernel before
  pdl_launch_dependents();
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float xv = x_last[i];
    ss += xv * xv;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[wid] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = rsqrtf(tot / static_cast<float>(d) + eps);
  for (int i = threadIdx.x; i < d; i += blockDim.x) hs[i] = x_last[i] * inv * __bfloat162float(g[i]);
  __syncthreads();
  unsigned long long mine = 0ull;
  for (; v < vocab; v += nwarps) {
    float acc = 0.f;
    // each lane sums its pieces in increasing order
    for (int it = 0; it < iters; ++it) {
      if (it > 0) issue(v, it);
#pragma unroll
      for (int u = 0; u < kLmLoads; ++u) {
        const int i = lane + 32 * (it * kLmLoads + u);
        if (i < n8) {
          float f[8];
          bf16x8_to_f32(wv[u], f);
          const float4 h0 = *reinterpret_cast<const float4*>(hs + 8 * i);
          const float4 h1 = *reinterpret_cast<const float4*>(hs + 8 * i + 4);
          acc += f[0] * h0.x + f[1] * h0.y + f[2] * h0.z + f[3] * h0.w + f[4] * h1.x + f[5] * h1.y + f[6] * h1.z +
                 f[7] * h1.w;
        }
      }
    }
    if (v + nwarps < vocab) issue(v + nwarps, 0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      logits[v] = acc;
      const unsigned long long k = argmax_key(acc, v);
      mine = k > mine ? k : mine;
    }
  }
  if (lane == 0) bred[wid] = mine;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long b = 0ull;
    for (int w = 0; w < 8; ++w) b = bred[w] > b ? bred[w] : b;
    best[blockIdx.x] = b;
  }
}

// One warp: the largest of the LM head's n per-CTA keys.
__global__ void argmax_finalize_kernel(const unsigned long long* best, int n, int32_t* token) {
  pdl_wait();
  unsigned long long b = 0ull;
  for (int i = threadIdx.x; i < n; i += 32) b = best[i] > b ? best[i] : b;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, b, o);
    b = y > b ? y : b;
  }
  if (threadIdx.x == 0) *token = static_cast<int32_t>(0xFFFFFFFFu - static_cast<unsigned int>(b & 0xFFFFFFFFull));
}

cudaError_t launch_embed(const __nv_bfloat16* embed, int vocab, int d, const int32_t* ids, const int32_t* rows,
                         int row_offset, int n, float* x, cudaStream_t st, bool pdl) {
  if (n <= 0) return cudaSuccess;
  LaunchScope ls(KC_EMBED, st);
  if (pdl)
    return launch_pdl(embed_rows_kernel, dim3((n + 7) / 8), dim3(256), 0, st, embed, vocab, d, ids, rows, row_offset,
                      n, x, device_status_ptr());
  embed_rows_kernel<<<(n + 7) / 8, 256, 0, st>>>(embed, vocab, d, ids, rows, row_offset, n, x, device_status_ptr());
  return cudaGetLastError();
}

// CTAs of the LM head: four per SM, at most kLmHeadSlots (one argmax key slot each).
constexpr int kLmHeadSlots = 4096;
static int lm_head_ctas() { return std::min(4 * num_sms(), kLmHeadSlots); }

cudaError_t launch_lm_head(const qcf_model* m, const float* x_last, float* logits, int32_t* token, void* best_ws,
                           cudaStream_t st, bool pdl) {
  unsigned long long* best = static_cast<unsigned long long*>(best_ws);
  const int d = m->dims.d_model, ctas = lm_head_ctas();
  const __nv_bfloat16* g = reinterpret_cast<const __nv_bfloat16*>(m->g_final);
  const __nv_bfloat16* W = reinterpret_cast<const __nv_bfloat16*>(m->lm_head);
  cudaError_t e;
  {
    LaunchScope ls(KC_LMHEAD, st);
    if (pdl) {
      e = launch_pdl(lm_head_kernel, dim3(ctas), dim3(256), d * sizeof(float), st, x_last, d, m->dims.vocab, g,
                     m->dims.eps, W, logits, best);
    } else {
      lm_head_kernel<<<ctas, 256, d * sizeof(float), st>>>(x_last, d, m->dims.vocab, g, m->dims.eps, W, logits, best);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
  }
  LaunchScope ls(KC_LMHEAD, st);
  return launch_pdl(argmax_finalize_kernel, dim3(1), dim3(32), 0, st, static_cast<const unsigned long long*>(best),
                    ctas, token);
}

cudaError_t launch_rmsnorm(const float* x, int n, int d, const __nv_bfloat16* g, float eps, __nv_bfloat16* h,
                           cudaStream_t st, bool pdl) {
  if (n <= 0) return cudaSuccess;
  LaunchScope ls(KC_RMSNORM, st);
  if (pdl) return launch_pdl(rmsnorm_kernel, dim3(n), dim3(kNormThreads), 0, st, x, n, d, g, eps, h);
  rmsnorm_kernel<<<n, kNormThreads, 0, st>>>(x, n, d, g, eps, h);
  return cudaGetLastError();
}

static qcf_status check_seg(const int32_t* seg_start, const int32_t* seg_delta, int n_seg, int64_t n_rows,
                            int max_pos, SegTable* t, const char* who) {
  if (n_seg <= 0 || n_seg > kMaxSeg) return set_error(QCF_ERR_SHAPE, "%s: n_seg=%d not in [1,%d]", who, n_seg, kMaxSeg);
  if (!seg_start || !seg_delta) return set_error(QCF_ERR_INVALID_ARG, "%s: segment table is NULL", who);
  if (seg_start[0] != 0 || seg_start[n_seg] != n_rows)
    return set_error(QCF_ERR_SHAPE, "%s: segments must cover [0, n_rows)", who);
  t->n_seg = n_seg;
  for (int s = 0; s <= n_seg; ++s) {
    if (s > 0 && seg_start[s] < seg_start[s - 1]) return set_error(QCF_ERR_SHAPE, "%s: seg_start not ascending", who);
    t->start[s] = seg_start[s];
  }
  for (int s = 0; s < n_seg; ++s) {
    if (seg_delta[s] < 0 || seg_delta[s] >= max_pos)
      return set_error(QCF_ERR_SHAPE, "%s: delta %d outside the RoPE table [0,%d)", who, seg_delta[s], max_pos);
    t->delta[s] = seg_delta[s];
  }
  return QCF_OK;
}

static bool head_dim_ok(int D) { return D == 16 || D == 64 || D == 128; }

cudaError_t launch_stage_scatter(const __nv_bfloat16* stK, const __nv_bfloat16* stV, const int32_t* src_row,
                                 const int32_t* delta, int64_t n_rows, int64_t staged_rows, int Hkv, int D,
                                 const qcf_rope_table* t, __nv_bfloat16* K, __nv_bfloat16* V, bool do_k, bool do_v,
                                 cudaStream_t st) {
  if (n_rows <= 0 || (!do_k && !do_v)) return cudaSuccess;
  const int64_t threads = n_rows * Hkv * (D / 16);
  LaunchScope ls(KC_ROPE, st);
  stage_scatter_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(
      stK, stV, src_row, delta, n_rows, staged_rows, Hkv, D, t->cos, t->sin, t->max_pos, K, V, do_k ? 1 : 0,
      do_v ? 1 : 0, device_status_ptr());
  return cudaGetLastError();
}

cudaError_t launch_reposition(const __nv_bfloat16* src, __nv_bfloat16* dst, int64_t n_rows, int Hkv, int D,
                              const int32_t* seg_start, const int32_t* seg_delta, int n_seg, const qcf_rope_table* t,
                              cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  SegTable seg;
  seg.n_seg = n_seg;
  for (int s = 0; s <= n_seg; ++s) seg.start[s] = seg_start[s];
  for (int s = 0; s < n_seg; ++s) seg.delta[s] = seg_delta[s];
  const int64_t threads = n_rows * Hkv * (D / 16);
  LaunchScope ls(KC_ROPE, st);
  rope_reposition_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(src, dst, n_rows, Hkv, D, t->cos,
                                                                                       t->sin, seg);
  return cudaGetLastError();
}

}  // namespace qcf

using namespace qcf;

extern "C" {

qcf_status qcf_rope_reposition(const qcf_bf16* K_src, qcf_bf16* K_dst, int64_t n_rows, int Hkv, int D,
                               const int32_t* seg_start, const int32_t* seg_delta, int n_seg,
                               const qcf_rope_table* t, void* stream) {
  if (!K_src || !K_dst || !t || !t->cos || !t->sin) return set_error(QCF_ERR_INVALID_ARG, "qcf_rope_reposition: NULL pointer");
  if (n_rows < 0 || Hkv <= 0 || !head_dim_ok(D) || t->head_dim != D)
    return set_error(QCF_ERR_SHAPE, "qcf_rope_reposition: n_rows=%lld Hkv=%d D=%d table D=%d", (long long)n_rows, Hkv, D,
                     t->head_dim);
  if (take_fault(4) || !aligned16(K_src) || !aligned16(K_dst) || !aligned16(t->cos) || !aligned16(t->sin))
    return set_error(QCF_ERR_ALIGN, "qcf_rope_reposition: pointers must be 16-byte aligned");
  SegTable seg;
  qcf_status s = check_seg(seg_start, seg_delta, n_seg, n_rows, t->max_pos, &seg, "qcf_rope_reposition");
  if (s != QCF_OK) return s;
  if (n_rows == 0) return QCF_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t threads = n_rows * Hkv * (D / 16);
  LaunchScope ls(KC_ROPE, st);
  rope_reposition_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(K_src), reinterpret_cast<__nv_bfloat16*>(K_dst), n_rows, Hkv, D, t->cos,
      t->sin, seg);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_rope_reposition: launch");
}

qcf_status qcf_gather_rows(const qcf_bf16* src, int64_t src_rows, int width, const int32_t* idx, int n, qcf_bf16* dst,
                           void* stream) {
  if (!src || !idx || !dst) return set_error(QCF_ERR_INVALID_ARG, "qcf_gather_rows: NULL pointer");
  if (n < 0 || src_rows < 0 || width <= 0 || width % 8)
    return set_error(QCF_ERR_SHAPE, "qcf_gather_rows: n=%d width=%d (width %% 8 == 0 required)", n, width);
  if (take_fault(4) || !aligned16(src) || !aligned16(dst)) return set_error(QCF_ERR_ALIGN, "qcf_gather_rows: alignment");
  if (take_fault(1)) return set_error(QCF_ERR_INVALID_ARG, "qcf_gather_rows: injected invalid index table");
  if (n == 0) return QCF_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LaunchScope ls(KC_GATHER, st);
  gather_rows_kernel<<<(n + 7) / 8, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), src_rows, width, idx, n,
                                                  reinterpret_cast<__nv_bfloat16*>(dst), device_status_ptr(),
                                                  check_enabled());
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_gather_rows: launch");
}

qcf_status qcf_scatter_kv(const qcf_bf16* k_new, const qcf_bf16* v_new, const int32_t* pos, int n, int Hkv, int D,
                          qcf_bf16* K_cache, qcf_bf16* V_cache, int T, void* stream) {
  if (!k_new || !v_new || !pos || !K_cache || !V_cache) return set_error(QCF_ERR_INVALID_ARG, "qcf_scatter_kv: NULL pointer");
  if (n < 0 || T < 0 || Hkv <= 0 || !head_dim_ok(D)) return set_error(QCF_ERR_SHAPE, "qcf_scatter_kv: bad shape");
  if (take_fault(4) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(K_cache) || !aligned16(V_cache))
    return set_error(QCF_ERR_ALIGN, "qcf_scatter_kv: alignment");
  if (take_fault(1)) return set_error(QCF_ERR_INVALID_ARG, "qcf_scatter_kv: injected invalid index table");
  if (n == 0) return QCF_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LaunchScope ls(KC_SCATTER, st);
  scatter_kv_kernel<<<(n + 7) / 8, 256, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16*>(k_new), reinterpret_cast<const __nv_bfloat16*>(v_new), pos, n, Hkv * D,
      reinterpret_cast<__nv_bfloat16*>(K_cache), reinterpret_cast<__nv_bfloat16*>(V_cache), T, device_status_ptr());
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_scatter_kv: launch");
}

qcf_status qcf_rmsnorm(const float* x, int n, int d, const qcf_bf16* g, float eps, qcf_bf16* h, void* stream) {
  if (!x || !g || !h) return set_error(QCF_ERR_INVALID_ARG, "qcf_rmsnorm: NULL pointer");
  if (n < 0 || d <= 0 || d % 8 || d > 8192)
    return set_error(QCF_ERR_SHAPE, "qcf_rmsnorm: d=%d must be a multiple of 8 and at most 8192", d);
  if (!aligned16(x) || !aligned16(g) || !aligned16(h)) return set_error(QCF_ERR_ALIGN, "qcf_rmsnorm: alignment");
  cudaError_t e = launch_rmsnorm(x, n, d, reinterpret_cast<const __nv_bfloat16*>(g), eps,
                                 reinterpret_cast<__nv_bfloat16*>(h), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_rmsnorm: launch");
}

qcf_status qcf_embed_rows(const qcf_model* m, const int32_t* ids, const int32_t* rows, int n, float* x, void* stream) {
  if (!m || !m->embed || !ids || !x) return set_error(QCF_ERR_INVALID_ARG, "qcf_embed_rows: NULL pointer");
  const int d = m->dims.d_model;
  if (n < 0 || d <= 0 || d % 8) return set_error(QCF_ERR_SHAPE, "qcf_embed_rows: bad shape");
  if (!aligned16(m->embed) || !aligned16(x)) return set_error(QCF_ERR_ALIGN, "qcf_embed_rows: alignment");
  if (n == 0) return QCF_OK;
  cudaError_t e = launch_embed(reinterpret_cast<const __nv_bfloat16*>(m->embed), m->dims.vocab, d, ids, rows, 0, n, x,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_embed_rows: launch");
}

size_t qcf_lm_head_workspace_size(const qcf_dims* dims) {
  (void)dims;
  return kLmHeadSlots * sizeof(unsigned long long);
}

qcf_status qcf_lm_head(const qcf_model* m, const float* x_last, float* logits, int32_t* token, void* ws,
                       size_t ws_bytes, void* stream) {
  if (!m || !m->lm_head || !m->g_final || !x_last || !logits || !token || !ws)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_lm_head: NULL pointer");
  if (ws_bytes < qcf_lm_head_workspace_size(&m->dims) || take_fault(2))
    return set_error(QCF_ERR_WORKSPACE, "qcf_lm_head: workspace too small");
  const int d = m->dims.d_model;
  if (d % 8 || d > 12288) return set_error(QCF_ERR_SHAPE, "qcf_lm_head: d=%d (at most 12288)", d);
  if (!aligned16(m->lm_head) || !aligned16(x_last)) return set_error(QCF_ERR_ALIGN, "qcf_lm_head: alignment");
  cudaError_t e = launch_lm_head(m, x_last, logits, token, ws, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_lm_head: launch");
}

}  // extern "C"
