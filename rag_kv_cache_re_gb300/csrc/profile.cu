// Critical-layer attention profiling: score[j] = sum_{r,h} softmax_j(scale q[r,h].K[j,g(h)]).
//
// The softmax of every (query row, head) is over all C context keys, so its
// normaliser is known only after a full pass over K.  Four launches:
//   pass 1  grid (key block, KV head, row group): per (row, head) running max and
//           sum of exp2 over the block's keys -> partial stats
//   merge   per (row, head): global max M and 1/L from the partials
//   pass 2  same grid: p = exp2(x - M) / L and column sums over the CTA's rows
//           -> one partial score vector per (KV head, row group)
//   sum     scores[j] = fixed-order sum of the partial vectors (deterministic)
// K tiles (64 keys) are staged by TMA through a 2-stage ring; Q.K^T runs on
// warp-level tensor cores (m16n8k16, fp32 accumulate).  Rows of a KV head's
// group are (head-in-group, query row) pairs; a CTA takes up to 256 of them
// (8 warps x 2 row tiles of 16).
#include <mutex>
#include <vector>

#include "qcf_internal.cuh"

namespace qcf {

constexpr int kPKeyTile = 64;
constexpr int kPRowsPerCta = 256;
constexpr int kPStages = 2;

template <int D>
__device__ __forceinline__ uint32_t ptile_off(int key, int col) {
  if constexpr (D >= 64) {
    return static_cast<uint32_t>((col >> 6) * (kPKeyTile * 128)) + sw128_off(key, (col & 63) >> 3);
  } else {
    return static_cast<uint32_t>(key * (D * 2) + col * 2);
  }
}

template <int D, bool PASS2>
__global__ void __launch_bounds__(256) profile_pass_kernel(const __grid_constant__ CUtensorMap tmK,
                                                           const __nv_bfloat16* __restrict__ q, int nq, int C, int Hq,
                                                           int G, int n_rg, int tiles_per_cta, float scale_log2,
                                                           float2* __restrict__ stats,
                                                           const float2* __restrict__ fstats,
                                                           float* __restrict__ part_scores, unsigned int* status) {
  constexpr int TILE_BYTES = kPKeyTile * D * 2;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPStages * TILE_BYTES);
  uint64_t* empty = full + kPStages;
  float* red = reinterpret_cast<float*>(empty + kPStages);  // [8][64] column sums (pass 2)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = blockIdx.x, g = blockIdx.y, rgi = blockIdx.z;
  const int R = nq * G;
  const int n_tiles_all = (C + kPKeyTile - 1) / kPKeyTile;
  const int t0 = kb * tiles_per_cta;
  const int t1 = min(n_tiles_all, t0 + tiles_per_cta);
  const int qc = (lane & 3) * 2;

  // this warp's two row tiles and the thread's four rows (lo/hi of each tile)
  int rho[2][2];
  bool rv[2][2];
  uint32_t qf[2][D / 16][4];
#pragma unroll
  for (int rt = 0; rt < 2; ++rt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      rho[rt][e] = rgi * kPRowsPerCta + (warp * 2 + rt) * 16 + (lane >> 2) + e * 8;
      rv[rt][e] = rho[rt][e] < R && (rho[rt][e] - rgi * kPRowsPerCta) < kPRowsPerCta;
    }
    const __nv_bfloat16* qp[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int rr = rv[rt][e] ? rho[rt][e] : 0;
      const int hh = rr / nq, r = rr - hh * nq;
      qp[e] = q + (static_cast<size_t>(r) * Hq + (g * G + hh)) * D;
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int k = ks * 16 + qc;
      qf[rt][ks][0] = rv[rt][0] ? *reinterpret_cast<const uint32_t*>(qp[0] + k) : 0u;
      qf[rt][ks][1] = rv[rt][1] ? *reinterpret_cast<const uint32_t*>(qp[1] + k) : 0u;
      qf[rt][ks][2] = rv[rt][0] ? *reinterpret_cast<const uint32_t*>(qp[0] + k + 8) : 0u;
      qf[rt][ks][3] = rv[rt][1] ? *reinterpret_cast<const uint32_t*>(qp[1] + k + 8) : 0u;
    }
  }
  const bool warp_active = rgi * kPRowsPerCta + warp * 32 < R;

  float m[2][2], l[2][2], fM[2][2], fI[2][2];
#pragma unroll
  for (int rt = 0; rt < 2; ++rt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      m[rt][e] = -INFINITY;
      l[rt][e] = 0.f;
      fM[rt][e] = 0.f;
      fI[rt][e] = 0.f;
      if (PASS2 && rv[rt][e]) {
        const int hh = rho[rt][e] / nq, r = rho[rt][e] - hh * nq;
        const float2 f = fstats[static_cast<size_t>(g * G + hh) * nq + r];
        fM[rt][e] = f.x;
        fI[rt][e] = f.y;
      }
    }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    fence_mbar_init();
  }
  __syncthreads();

  constexpr int boxes = D >= 64 ? D / 64 : 1;
  constexpr int box_cols = D >= 64 ? 64 : D;
  auto issue = [&](int t) {
    const int s = (t - t0) % kPStages;
    uint8_t* kbuf = smem + s * TILE_BYTES;
    mbar_arrive_expect_tx(&full[s], TILE_BYTES);
#pragma unroll
    for (int b = 0; b < boxes; ++b)
      tma_load_2d(kbuf + b * kPKeyTile * box_cols * 2, &tmK, &full[s], g * D + b * box_cols, t * kPKeyTile);
  };
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    for (int t = t0; t < t1 && t < t0 + kPStages; ++t) issue(t);
  }

  bool ok = true;
  for (int t = t0; t < t1; ++t) {
    const int it = t - t0;
    const int s = it % kPStages;
    const uint32_t par = (it / kPStages) & 1;
    const bool got = mbar_wait(&full[s], par);
    if (!got) flag_status(status, QCF_DEV_TIMEOUT);
    if (PASS2) {
      // pass 2 has block barriers below: give up only when the whole CTA agrees
      if (__syncthreads_or(!got)) return;
    } else if (!got) {
      ok = false;
      break;
    }
    const int j0 = t * kPKeyTile;
    float colsum[8][2];
#pragma unroll
    for (int i = 0; i < 8; ++i) colsum[i][0] = colsum[i][1] = 0.f;
    if (warp_active) {
      const uint32_t kaddr = smem_u32(smem + s * TILE_BYTES);
      float sc[2][8][4];
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[rt][i][0] = sc[rt][i][1] = sc[rt][i][2] = sc[rt][i][3] = 0.f;
      const int mi = lane >> 3, mr = lane & 7;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kaddr + ptile_off<D>(np * 16 + (mi >> 1) * 8 + mr, ks * 16 + (mi & 1) * 8), b0, b1, b2, b3);
#pragma unroll
          for (int rt = 0; rt < 2; ++rt) {
            mma_bf16_16816(sc[rt][2 * np], qf[rt][ks], b0, b1);
            mma_bf16_16816(sc[rt][2 * np + 1], qf[rt][ks], b2, b3);
          }
        }
      }
#pragma unroll
      for (int rt = 0; rt < 2; ++rt) {
        if (!PASS2) {
          float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = j0 + nt * 8 + qc + (e & 1);
              const float x = key < C ? sc[rt][nt][e] * scale_log2 : -INFINITY;
              sc[rt][nt][e] = x;
              tmax[e >> 1] = fmaxf(tmax[e >> 1], x);
            }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mn = fmaxf(m[rt][e], tmax[e]);
            const float base = mn == -INFINITY ? 0.f : mn;
            float acc = l[rt][e] * exp2f(m[rt][e] - base);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) acc += exp2f(sc[rt][nt][2 * e] - base) + exp2f(sc[rt][nt][2 * e + 1] - base);
            l[rt][e] = acc;
            m[rt][e] = mn;
          }
        } else {
#pragma unroll
          for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = j0 + nt * 8 + qc + (e & 1);
              const int re = e >> 1;
              const float p = (key < C && rv[rt][re]) ? exp2f(sc[rt][nt][e] * scale_log2 - fM[rt][re]) * fI[rt][re] : 0.f;
              colsum[nt][e & 1] += p;
            }
        }
      }
    }
    if (PASS2) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = colsum[nt][e];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          colsum[nt][e] = v;
        }
      if (lane < 4) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          red[warp * 64 + nt * 8 + qc] = colsum[nt][0];
          red[warp * 64 + nt * 8 + qc + 1] = colsum[nt][1];
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (PASS2) {
      __syncthreads();
      if (threadIdx.x < 64) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) v += red[w * 64 + threadIdx.x];
        const int key = j0 + threadIdx.x;
        if (key < C) part_scores[static_cast<size_t>(g * n_rg + rgi) * C + key] = v;
      }
      __syncthreads();
    }
    if (warp == 0) {
      if (lane == 0 && t + kPStages < t1) {
        if (!mbar_wait(&empty[s], par)) {
          // nothing more is issued: every thread's next full-barrier wait runs out
          flag_status(status, QCF_DEV_TIMEOUT);
          if (!PASS2) ok = false;
        } else {
          issue(t + kPStages);
        }
      }
      __syncwarp();
    }
    if (!ok) break;
  }
  if (!ok) return;

  if (!PASS2) {
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mm = m[rt][e], ll = l[rt][e];
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
          const float om = __shfl_xor_sync(0xffffffffu, mm, o);
          const float ol = __shfl_xor_sync(0xffffffffu, ll, o);
          const float mn = fmaxf(mm, om);
          const float base = mn == -INFINITY ? 0.f : mn;
          ll = ll * exp2f(mm - base) + ol * exp2f(om - base);
          mm = mn;
        }
        if ((lane & 3) == 0 && rv[rt][e]) {
          const int hh = rho[rt][e] / nq, r = rho[rt][e] - hh * nq;
          stats[static_cast<size_t>(kb) * Hq * nq + static_cast<size_t>(g * G + hh) * nq + r] = make_float2(mm, ll);
        }
      }
  }
}

// Per (head, row): M = max of the partial maxima, L = sum l_i 2^(m_i - M); writes (M, 1/L).
__global__ void profile_merge_kernel(const float2* __restrict__ stats, int n_kb, int rows, float2* __restrict__ fstats) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows) return;
  float M = -INFINITY;
  for (int k = 0; k < n_kb; ++k) M = fmaxf(M, stats[static_cast<size_t>(k) * rows + i].x);
  float L = 0.f;
  for (int k = 0; k < n_kb; ++k) {
    const float2 s = stats[static_cast<size_t>(k) * rows + i];
    if (s.y > 0.f) L += s.y * exp2f(s.x - M);
  }
  fstats[i] = make_float2(M, L > 0.f ? 1.f / L : 0.f);
}

// scores[j] = sum over the P partial vectors in index order.
__global__ void profile_sum_kernel(const float* __restrict__ part, int P, int C, float* __restrict__ scores) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= C) return;
  float v = 0.f;
  for (int p = 0; p < P; ++p) v += part[static_cast<size_t>(p) * C + j];
  scores[j] = v;
}

struct ProfilePlan {
  int n_rg, n_tiles, tpc, n_kb;
  size_t stats_bytes, fstats_bytes, part_bytes;
};

static ProfilePlan plan_profile(int nq, int C, int Hq, int Hkv) {
  ProfilePlan p;
  const int G = Hq / Hkv;
  p.n_rg = (nq * G + kPRowsPerCta - 1) / kPRowsPerCta;
  p.n_tiles = (C + kPKeyTile - 1) / kPKeyTile;
  const int sms = num_sms();
  const int target_kb = (4 * sms + Hkv * p.n_rg - 1) / (Hkv * p.n_rg);
  p.tpc = (p.n_tiles + target_kb - 1) / (target_kb > 0 ? target_kb : 1);
  if (p.tpc < 1) p.tpc = 1;
  p.n_kb = (p.n_tiles + p.tpc - 1) / p.tpc;
  p.stats_bytes = align_up(static_cast<size_t>(p.n_kb) * Hq * nq * sizeof(float2), 256);
  p.fstats_bytes = align_up(static_cast<size_t>(Hq) * nq * sizeof(float2), 256);
  p.part_bytes = align_up(static_cast<size_t>(Hkv) * p.n_rg * C * sizeof(float), 256);
  return p;
}

template <int D>
static qcf_status profile_launch_d(const __nv_bfloat16* q, const __nv_bfloat16* K, int nq, int C, int Hq, int Hkv,
                                   float scale, float* scores, void* ws, cudaStream_t st) {
  const ProfilePlan p = plan_profile(nq, C, Hq, Hkv);
  float2* stats = static_cast<float2*>(ws);
  float2* fstats = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + p.stats_bytes);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + p.stats_bytes + p.fstats_bytes);
  CUtensorMap tk;
  const uint64_t width = static_cast<uint64_t>(Hkv) * D;
  const uint32_t box_cols = D >= 64 ? 64 : D;
  if (!encode_tmap_2d(&tk, K, width, C, width * 2, box_cols, kPKeyTile,
                      D >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE))
    return set_error(QCF_ERR_CUDA, "profile_scores: tensor map encoding failed");
  const int smem = kPStages * kPKeyTile * D * 2 + 64 + 8 * 64 * 4 + 1024;
  static PerDevice<cudaError_t> smem_attr;
  const cudaError_t attr = smem_attr.get(current_device(), [smem] {
    cudaError_t e = cudaFuncSetAttribute(profile_pass_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(profile_pass_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return e;
  });
  if (attr != cudaSuccess) return cuda_error(attr, "profile_scores: smem attribute");
  const int G = Hq / Hkv;
  const float scale_log2 = scale * 1.4426950408889634f;
  dim3 grid(p.n_kb, Hkv, p.n_rg);
  unsigned int* status = device_status_ptr();
  {
    LaunchScope ls(KC_PROFILE, st);
    profile_pass_kernel<D, false><<<grid, 256, smem, st>>>(tk, q, nq, C, Hq, G, p.n_rg, p.tpc, scale_log2, stats,
                                                           nullptr, nullptr, status);
  }
  const int rows = Hq * nq;
  {
    LaunchScope ls(KC_PROFILE, st);
    profile_merge_kernel<<<(rows + 255) / 256, 256, 0, st>>>(stats, p.n_kb, rows, fstats);
  }
  {
    LaunchScope ls(KC_PROFILE, st);
    profile_pass_kernel<D, true><<<grid, 256, smem, st>>>(tk, q, nq, C, Hq, G, p.n_rg, p.tpc, scale_log2, nullptr,
                                                          fstats, part, status);
  }
  {
    LaunchScope ls(KC_PROFILE, st);
    profile_sum_kernel<<<(C + 255) / 256, 256, 0, st>>>(part, Hkv * p.n_rg, C, scores);
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "profile_scores: launch");
}

// ------------------------------------------------------------------ fixed scratch for callers that cannot allocate
//
// Scratch of qcf_profile_scores_noalloc: one array in device global memory that
// exists for the life of the process on every GPU that loads this library.  Its
// contents persist between calls; every call fully rewrites the parts it reads,
// so nothing in it has to start at zero.
constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_profile_scratch[kNoAllocScratchBytes];

// Device address of g_profile_scratch for the current device, looked up once per
// device (the symbol name is a host-side stand-in, not an address a kernel may use).
static qcf_status profile_scratch_address(void** out) {
  static std::mutex mu;
  static std::vector<void*> per_dev;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "qcf_profile_scores_noalloc: cudaGetDevice");
  std::lock_guard<std::mutex> lk(mu);
  if (static_cast<int>(per_dev.size()) <= dev) per_dev.resize(dev + 1, nullptr);
  if (!per_dev[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_profile_scratch);
    if (e != cudaSuccess) return cuda_error(e, "qcf_profile_scores_noalloc: cudaGetSymbolAddress");
    per_dev[dev] = p;
  }
  *out = per_dev[dev];
  return QCF_OK;
}

}  // namespace qcf

using namespace qcf;

extern "C" {

static bool use_tc_profile(int Hq, int Hkv, int D) { return D == 128 && Hq / Hkv <= kProfileTcMaxGroup; }

size_t qcf_profile_scores_workspace_size(int nq, int C, int Hq, int Hkv, int D) {
  if (nq <= 0 || C <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return 0;
  if (use_tc_profile(Hq, Hkv, D)) return profile_tc_workspace_size(nq, C, Hq, Hkv);
  const ProfilePlan p = plan_profile(nq, C, Hq, Hkv);
  return p.stats_bytes + p.fstats_bytes + p.part_bytes;
}

qcf_status qcf_profile_scores(const qcf_bf16* q, const qcf_bf16* K, int nq, int C, int Hq, int Hkv, int D, float scale,
                              float* scores, void* ws, size_t ws_bytes, void* stream) {
  if (!q || !K || !scores || !ws) return set_error(QCF_ERR_INVALID_ARG, "qcf_profile_scores: NULL pointer");
  if (nq <= 0 || C <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || (D != 16 && D != 64 && D != 128))
    return set_error(QCF_ERR_SHAPE, "qcf_profile_scores: nq=%d C=%d Hq=%d Hkv=%d D=%d", nq, C, Hq, Hkv, D);
  if (!(scale > 0.f) || !isfinite(scale))
    return set_error(QCF_ERR_INVALID_ARG, "qcf_profile_scores: scale must be positive and finite");
  if (take_fault(4) || !aligned16(q) || !aligned16(K) || !aligned16(scores) || !aligned16(ws))
    return set_error(QCF_ERR_ALIGN, "qcf_profile_scores: pointers must be 16-byte aligned");
  if (take_fault(2) || ws_bytes < qcf_profile_scores_workspace_size(nq, C, Hq, Hkv, D))
    return set_error(QCF_ERR_WORKSPACE, "qcf_profile_scores: workspace %zu < %zu", ws_bytes,
                     qcf_profile_scores_workspace_size(nq, C, Hq, Hkv, D));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* qq = reinterpret_cast<const __nv_bfloat16*>(q);
  const __nv_bfloat16* kk = reinterpret_cast<const __nv_bfloat16*>(K);
  if (use_tc_profile(Hq, Hkv, D)) return profile_tc_launch(qq, kk, nq, C, Hq, Hkv, scale, scores, ws, st);
  switch (D) {
    case 16: return profile_launch_d<16>(qq, kk, nq, C, Hq, Hkv, scale, scores, ws, st);
    case 64: return profile_launch_d<64>(qq, kk, nq, C, Hq, Hkv, scale, scores, ws, st);
    default: return profile_launch_d<128>(qq, kk, nq, C, Hq, Hkv, scale, scores, ws, st);
  }
}

qcf_status qcf_profile_scores_noalloc(const qcf_bf16* q, const qcf_bf16* K, int nq, int C, int Hq, int Hkv, int D,
                                      float scale, float* scores, void* stream) {
  if (!q || !K || !scores) return set_error(QCF_ERR_INVALID_ARG, "qcf_profile_scores_noalloc: NULL pointer");
  if (nq <= 0 || C <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || (D != 16 && D != 64 && D != 128))
    return set_error(QCF_ERR_SHAPE, "qcf_profile_scores_noalloc: nq=%d C=%d Hq=%d Hkv=%d D=%d", nq, C, Hq, Hkv, D);
  if (!(scale > 0.f) || !isfinite(scale))
    return set_error(QCF_ERR_INVALID_ARG, "qcf_profile_scores_noalloc: scale must be positive and finite");
  if (!aligned16(q) || !aligned16(K) || !aligned16(scores))
    return set_error(QCF_ERR_ALIGN, "qcf_profile_scores_noalloc: pointers must be 16-byte aligned");
  const size_t need = qcf_profile_scores_workspace_size(nq, C, Hq, Hkv, D);
  if (need > kNoAllocScratchBytes)
    return set_error(QCF_ERR_WORKSPACE,
                     "qcf_profile_scores_noalloc: this shape needs %zu bytes of scratch, more than the fixed %zu; "
                     "use qcf_profile_scores with a caller workspace",
                     need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  qcf_status st = profile_scratch_address(&scratch);
  if (st != QCF_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* qq = reinterpret_cast<const __nv_bfloat16*>(q);
  const __nv_bfloat16* kk = reinterpret_cast<const __nv_bfloat16*>(K);
  if (use_tc_profile(Hq, Hkv, D)) return profile_tc_launch(qq, kk, nq, C, Hq, Hkv, scale, scores, scratch, cs);
  switch (D) {
    case 16: return profile_launch_d<16>(qq, kk, nq, C, Hq, Hkv, scale, scores, scratch, cs);
    case 64: return profile_launch_d<64>(qq, kk, nq, C, Hq, Hkv, scale, scores, scratch, cs);
    default: return profile_launch_d<128>(qq, kk, nq, C, Hq, Hkv, scale, scores, scratch, cs);
  }
}

}  // extern "C"
