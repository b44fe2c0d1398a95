// Critical-layer attention profiling on the 5th-generation tensor cores (head dim 128):
// score[j] = sum over query rows r and heads h of softmax_j(scale * q[r,h] . K[j, h / G]).
//
// Every (row, head) softmax runs over all C context keys, so its normaliser is known
// only after a full pass over K: two kernels, each streaming K once.
//   pass 1  CTA (key chunk, KV head g, row group): per score row (a query row and one of
//           the G heads of g) the running max and sum of exp2 over the chunk's keys;
//           S = Q K^T with the score rows in TMEM lanes, one thread per row.
//   pass 2  the same grid, launched programmatically behind pass 1: each CTA first merges
//           its rows' partial statistics into M' = M + log2(L), then computes the
//           transposed S^T = K Q^T with the keys in TMEM lanes, one thread per key, and sums
//           exp2(scale' s - M') over the CTA's rows inside the thread.  The last CTA of a
//           key chunk to finish adds the chunk's partial vectors in a fixed order (the
//           result is the same bits on every run) and writes the scores.
// K tiles of 128 keys (two 64-column boxes, 128-byte swizzle) stream by TMA through a
// 4-stage ring; the CTA's query rows (up to two row tiles of 128) stay in shared memory,
// loaded once by a rank-3 TMA box over (head dim, head, query row).  One thread issues
// the tensor-core work into a double-buffered TMEM accumulator; pass 2 walks its chunk in
// reverse so its first tiles are the ones pass 1 read last, still in L2.
#include "qcf_internal.cuh"

namespace qcf {

constexpr int kPtKeys = 128;
constexpr int kPtStages = 4;
constexpr int kPtThreads = 320;                       // producer, MMA, 8 softmax warps
constexpr int kPtBoxBytes = kPtKeys * 128;            // 128 keys x 64 bf16
constexpr int kPtTileBytes = 2 * kPtBoxBytes;         // 128 keys x 128 bf16
constexpr int kPtQBytes = 4 * 128 * 128;              // 2 row tiles x 2 column boxes x 128 rows x 64 bf16
constexpr int kPtSmem = kPtQBytes + kPtStages * kPtTileBytes + 4096 + 1024;

struct ProfileTcPlan {
  int G, R, RT;        // heads per KV head, query rows per row tile, score rows per row tile (R * G <= 128)
  int n_rt, n_rg;      // row tiles per KV head, row groups (two row tiles each)
  int n_tiles, tpc, n_kc;
  size_t stats_bytes, part_bytes, cnt_bytes;
};

static ProfileTcPlan plan_profile_tc(int nq, int C, int Hq, int Hkv) {
  ProfileTcPlan p;
  p.G = Hq / Hkv;
  p.R = 128 / p.G;
  p.RT = p.R * p.G;
  p.n_rt = (nq + p.R - 1) / p.R;
  p.n_rg = (p.n_rt + 1) / 2;
  p.n_tiles = (C + kPtKeys - 1) / kPtKeys;
  int kc = num_sms() / (Hkv * p.n_rg);
  if (kc < 1) kc = 1;
  if (kc > p.n_tiles) kc = p.n_tiles;
  p.tpc = (p.n_tiles + kc - 1) / kc;
  p.n_kc = (p.n_tiles + p.tpc - 1) / p.tpc;
  p.stats_bytes = align_up(static_cast<size_t>(Hkv) * p.n_rg * p.n_kc * 256 * sizeof(float2), 256);
  p.part_bytes = align_up(static_cast<size_t>(Hkv) * p.n_rg * C * sizeof(float), 256);
  p.cnt_bytes = align_up(static_cast<size_t>(p.n_kc) * sizeof(unsigned int), 256);
  return p;
}

size_t profile_tc_workspace_size(int nq, int C, int Hq, int Hkv) {
  const ProfileTcPlan p = plan_profile_tc(nq, C, Hq, Hkv);
  return p.stats_bytes + p.part_bytes + p.cnt_bytes;
}

template <bool PASS2>
__global__ void __launch_bounds__(kPtThreads, 1)
    profile_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ, int nq, int C,
                      int G, int R, int RT, int n_rt, int n_rg, int tpc, int n_kc, float scale_log2,
                      float2* __restrict__ stats, float* __restrict__ part, unsigned int* __restrict__ counters,
                      float* __restrict__ scores, unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* qbuf = smem;                     // box (column half hb, row tile t) at hb * 32 KB + t * 16 KB
  uint8_t* kbuf = smem + kPtQBytes;         // stage st at st * 32 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(kbuf + kPtStages * kPtTileBytes);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + kPtStages;
  uint64_t* s_full = k_empty + kPtStages;
  uint64_t* s_free = s_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_free + 2);
  uint32_t* last_flag = tmem_slot + 1;
  float* mp = reinterpret_cast<float*>(smem + kPtQBytes + kPtStages * kPtTileBytes + 1024);   // [2][128] M' (pass 2)
  float* red = mp + 256;                                                                      // [2][128] (pass 2)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kc = blockIdx.x, g = blockIdx.y, rg = blockIdx.z;
  const int n_tiles = (C + kPtKeys - 1) / kPtKeys;
  const int t0 = kc * tpc;
  const int t1 = min(n_tiles, t0 + tpc);
  const int nt = t1 - t0;  // >= 1 by the plan
  const int n_rt_cta = min(2, n_rt - rg * 2);
  const int n_part = gridDim.y * n_rg;

  if (!PASS2) {
    pdl_launch_dependents();
    if (kc == 0 && g == 0 && rg == 0)
      for (int i = threadIdx.x; i < n_kc; i += blockDim.x) counters[i] = 0u;
  }
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kPtStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 4 * n_rt_cta);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (RT < 128) {
    // rows RT..127 of each query row tile lie outside the TMA boxes: zero them, so the
    // transposed scores of pass 2 hold zeros (not stale bits) in those columns
    const int pad = (128 - RT) * 128 / 16;  // 16-byte words per box
    for (int w = threadIdx.x; w < 4 * pad; w += blockDim.x) {
      const int box = w / pad, k = w - box * pad;
      *reinterpret_cast<uint4*>(qbuf + (box >> 1) * 32768 + (box & 1) * 16384 + RT * 128 + k * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer: the CTA's query rows once, then the chunk's K tiles
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmQ);
      mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(n_rt_cta * 2 * RT * 128));
      for (int t = 0; t < n_rt_cta; ++t)
#pragma unroll
        for (int hb = 0; hb < 2; ++hb)
          tma_load_3d(qbuf + hb * 32768 + t * 16384, &tmQ, q_full, hb * 64, g * G, (rg * 2 + t) * R);
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int st = i % kPtStages;
        if (!mbar_wait(&k_empty[st], ((i / kPtStages) & 1) ^ 1u)) {
          flag_status(status, QCF_DEV_TIMEOUT);
          break;
        }
        const int tk = PASS2 ? t1 - 1 - i : t0 + i;
        mbar_arrive_expect_tx(&k_full[st], kPtTileBytes);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb)
          tma_load_2d(kbuf + st * kPtTileBytes + hb * kPtBoxBytes, &tmK, &k_full[st], g * 128 + hb * 64, tk * kPtKeys);
        ++issued;
      }
      // no copy may still be landing in this CTA's shared memory when it exits
      for (int i = max(0, issued - kPtStages); i < issued; ++i)
        if (!mbar_wait(&k_full[i % kPtStages], (i / kPtStages) & 1)) flag_status(status, QCF_DEV_TIMEOUT);
      if (!mbar_wait(q_full, 0)) flag_status(status, QCF_DEV_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = smem_u32(qbuf), k_addr = smem_u32(kbuf);
      const uint32_t idesc_s = idesc_bf16_f32(128, kPtKeys);           // pass 1: rows x keys
      const uint32_t idesc_t = idesc_bf16_f32(128, 128 * n_rt_cta);    // pass 2: keys x rows
      bool ok = mbar_wait(q_full, 0);
      int done = 0;
      for (int i = 0; i < nt && ok; ++i) {
        const int st = i % kPtStages, b = i & 1;
        if (!mbar_wait(&k_full[st], (i / kPtStages) & 1) || !mbar_wait(&s_free[b], ((i >> 1) & 1) ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kst = k_addr + st * kPtTileBytes;
        if (!PASS2) {
          for (int t = 0; t < n_rt_cta; ++t)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_f16(tmem_base + b * 256 + t * 128,
                       sdesc_kmajor_sw128(q_addr + (kk >> 2) * 32768 + t * 16384 + (kk & 3) * 32),
                       sdesc_kmajor_sw128(kst + (kk >> 2) * kPtBoxBytes + (kk & 3) * 32), idesc_s, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_f16(tmem_base + b * 256, sdesc_kmajor_sw128(kst + (kk >> 2) * kPtBoxBytes + (kk & 3) * 32),
                     sdesc_kmajor_sw128(q_addr + (kk >> 2) * 32768 + (kk & 3) * 32), idesc_t, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[b]);
        umma_commit(&k_empty[st]);
        done = i + 1;
      }
      if (!ok) flag_status(status, QCF_DEV_TIMEOUT);
      // the last issued tile's MMAs and both of their barrier arrivals are complete before
      // tensor memory is freed and the CTA's shared memory is released
      if (done > 0 && (!mbar_wait(&s_full[(done - 1) & 1], ((done - 1) >> 1) & 1) ||
                       !mbar_wait(&k_empty[(done - 1) % kPtStages], ((done - 1) / kPtStages) & 1)))
        flag_status(status, QCF_DEV_TIMEOUT);
    }
  } else {
    // ---- softmax warps: warpgroup wg serves row tile wg; TMEM lanes by warp % 4
    constexpr unsigned kAll = 0xffffffffu;
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int l128 = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const bool active = wg < n_rt_cta;
    const size_t part_row = static_cast<size_t>(g * n_rg + rg);
    if (!PASS2) {
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < nt && active; ++i) {
        const int b = i & 1;
        if (!__all_sync(kAll, mbar_wait(&s_full[b], (i >> 1) & 1))) {
          flag_status(status, QCF_DEV_TIMEOUT);
          break;
        }
        tc_fence_after();
        float v[128];
        tmem_ld64(tmem_base + lane_base + b * 256 + wg * 128, v);
        tmem_ld64(tmem_base + lane_base + b * 256 + wg * 128 + 64, v + 64);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[b]);
        const int j0 = (t0 + i) * kPtKeys;
        if (j0 + kPtKeys > C) {
#pragma unroll
          for (int k = 0; k < kPtKeys; ++k)
            if (j0 + k >= C) v[k] = -INFINITY;
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const float* w = v + h2 * 64;
          float a0 = w[0], a1 = w[1], a2 = w[2], a3 = w[3];
#pragma unroll
          for (int k = 4; k < 64; k += 4) {
            a0 = fmaxf(a0, w[k]);
            a1 = fmaxf(a1, w[k + 1]);
            a2 = fmaxf(a2, w[k + 2]);
            a3 = fmaxf(a3, w[k + 3]);
          }
          const float mn = fmaxf(m, fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * scale_log2);
          const float base = mn == -INFINITY ? 0.f : mn;
          const float nb = -base;
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int k = 0; k < 64; k += 4) {
            s0 += fast_exp2(fmaf(w[k], scale_log2, nb));
            s1 += fast_exp2(fmaf(w[k + 1], scale_log2, nb));
            s2 += fast_exp2(fmaf(w[k + 2], scale_log2, nb));
            s3 += fast_exp2(fmaf(w[k + 3], scale_log2, nb));
          }
          l = l * fast_exp2(m - base) + ((s0 + s1) + (s2 + s3));
          m = mn;
        }
      }
      if (active) {
        const size_t o = (part_row * n_kc + kc) * 256 + wg * 128 + l128;
        stats[o] = make_float2(m, l);
      }
    } else {
      pdl_wait();  // the statistics of pass 1
      // M' = M + log2(L) of this thread's row; rows past the query or in the padding of a
      // row tile get +inf, which zeroes their terms
      {
        float Mp = INFINITY;
        const int r = (rg * 2 + wg) * R + l128 / G;
        if (active && l128 < RT && r < nq) {
          float M = -INFINITY;
          for (int k = 0; k < n_kc; ++k) M = fmaxf(M, stats[(part_row * n_kc + k) * 256 + wg * 128 + l128].x);
          float L = 0.f;
          for (int k = 0; k < n_kc; ++k) {
            const float2 sv = stats[(part_row * n_kc + k) * 256 + wg * 128 + l128];
            if (sv.y > 0.f) L += sv.y * exp2f(sv.x - M);
          }
          if (L > 0.f) Mp = M + log2f(L);
        }
        mp[wg * 128 + l128] = Mp;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      bool ok = true;
      for (int i = 0; i < nt; ++i) {
        const int b = i & 1;
        const int tk = t1 - 1 - i;
        float acc = 0.f;
        if (active) {
          if (!__all_sync(kAll, mbar_wait(&s_full[b], (i >> 1) & 1))) {
            flag_status(status, QCF_DEV_TIMEOUT);
            ok = false;
          }
          if (ok) {
            tc_fence_after();
            float v[128];
            tmem_ld64(tmem_base + lane_base + b * 256 + wg * 128, v);
            tmem_ld64(tmem_base + lane_base + b * 256 + wg * 128 + 64, v + 64);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[b]);
            const float4* m4 = reinterpret_cast<const float4*>(mp + wg * 128);
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const float4 mm = m4[k];
              s0 += fast_exp2(fmaf(v[4 * k], scale_log2, -mm.x));
              s1 += fast_exp2(fmaf(v[4 * k + 1], scale_log2, -mm.y));
              s2 += fast_exp2(fmaf(v[4 * k + 2], scale_log2, -mm.z));
              s3 += fast_exp2(fmaf(v[4 * k + 3], scale_log2, -mm.w));
            }
            acc = (s0 + s1) + (s2 + s3);
          }
        }
        // a timed-out warp leaves the loop with every other softmax warp (no barrier waits on it)
        if (bar_red_or(1, 256, !ok)) break;
        if (n_rt_cta > 1) {
          if (wg == 1) red[(i & 1) * 128 + l128] = acc;
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (wg == 0) acc += red[(i & 1) * 128 + l128];
        }
        const int j = tk * kPtKeys + l128;
        if (wg == 0 && j < C) part[part_row * C + j] = acc;
      }
      // the last of the chunk's CTAs to finish adds the n_part partial vectors in order
      __threadfence();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (warp == 2 && lane == 0) {
        const unsigned int prev = atomicAdd(&counters[kc], 1u);
        *last_flag = prev == static_cast<unsigned int>(n_part - 1) ? 1u : 0u;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (*last_flag) {
        __threadfence();
        const int j_end = min(C, t1 * kPtKeys);
        for (int j = t0 * kPtKeys + (threadIdx.x - 64); j < j_end; j += 256) {
          float s = 0.f;
          for (int p = 0; p < n_part; ++p) s += __ldcg(part + static_cast<size_t>(p) * C + j);
          scores[j] = s;
        }
        if (warp == 2 && lane == 0) counters[kc] = 0u;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

qcf_status profile_tc_launch(const __nv_bfloat16* q, const __nv_bfloat16* K, int nq, int C, int Hq, int Hkv,
                             float scale, float* scores, void* ws, cudaStream_t st) {
  const ProfileTcPlan p = plan_profile_tc(nq, C, Hq, Hkv);
  float2* stats = static_cast<float2*>(ws);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + p.stats_bytes);
  unsigned int* cnt = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + p.stats_bytes + p.part_bytes);
  CUtensorMap tk, tq;
  const uint64_t width = static_cast<uint64_t>(Hkv) * 128;
  if (!encode_tmap_2d(&tk, K, width, C, width * 2, 64, kPtKeys, CU_TENSOR_MAP_SWIZZLE_128B))
    return set_error(QCF_ERR_CUDA, "profile_scores: K tensor map encoding failed");
  const uint64_t qdims[3] = {128, static_cast<uint64_t>(Hq), static_cast<uint64_t>(nq)};
  const uint64_t qstrides[2] = {128 * 2, static_cast<uint64_t>(Hq) * 128 * 2};
  const uint32_t qbox[3] = {64, static_cast<uint32_t>(p.G), static_cast<uint32_t>(p.R)};
  if (!encode_tmap_3d(&tq, q, qdims, qstrides, qbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return set_error(QCF_ERR_CUDA, "profile_scores: q tensor map encoding failed");
  static PerDevice<cudaError_t> smem_attr;
  const cudaError_t attr = smem_attr.get(current_device(), [] {
    cudaError_t e = cudaFuncSetAttribute(profile_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPtSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(profile_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPtSmem);
    return e;
  });
  if (attr != cudaSuccess) return cuda_error(attr, "profile_scores: smem attribute");
  const float scale_log2 = scale * 1.4426950408889634f;
  const dim3 grid(p.n_kc, Hkv, p.n_rg);
  unsigned int* status = device_status_ptr();
  {
    LaunchScope ls(KC_PROFILE, st);
    profile_tc_kernel<false><<<grid, kPtThreads, kPtSmem, st>>>(tk, tq, nq, C, p.G, p.R, p.RT, p.n_rt, p.n_rg, p.tpc,
                                                               p.n_kc, scale_log2, stats, part, cnt, scores, status);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "profile_scores: pass 1 launch");
  {
    LaunchScope ls(KC_PROFILE, st);
    e = launch_pdl(profile_tc_kernel<true>, grid, dim3(kPtThreads), kPtSmem, st, tk, tq, nq, C, p.G, p.R, p.RT, p.n_rt,
                   p.n_rg, p.tpc, p.n_kc, scale_log2, stats, part, cnt, scores, status);
  }
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "profile_scores: pass 2 launch");
}

}  // namespace qcf
