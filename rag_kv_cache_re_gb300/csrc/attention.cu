// Location-aware sparse causal attention over the fused KV cache.
//
// Recomputed rows arrive sorted by their absolute position.  A CTA takes a block
// of BR consecutive rows and one KV head g with all G = Hq/Hkv query heads that
// share it; warp w handles 16 rows of query head g*G + (w % G).  The CTA streams
// K/V tiles of 64 keys from 0 up to the largest position of its rows (rows are
// ascending, so that is its last row's position) through a 2-stage TMA ring; each
// warp skips tiles beyond its own rows and masks keys j > pos inside the
// boundary tiles.  Q.K^T and P.V run on warp-level tensor cores (m16n8k16, bf16
// in, fp32 accumulate); the softmax is online in fp32 registers with quad
// shuffles for the row max.  Blocks are scheduled longest (highest position)
// first.
#include <algorithm>
#include <mutex>

#include "qcf_internal.cuh"

namespace qcf {

constexpr int kKeyTile = 64;
constexpr int kAttnStages = 2;

template <int D>
struct AttnCfg {
  static constexpr int TILE_BYTES = kKeyTile * D * 2;  // one of K or V
  static constexpr int SMEM_BYTES = kAttnStages * 2 * TILE_BYTES + 256 + 1024;
  static constexpr bool SW128 = D >= 64;
};

// Byte offset of element (key, col) in a K or V tile; col % 8 == 0.
template <int D>
__device__ __forceinline__ uint32_t tile_off(int key, int col) {
  if constexpr (D >= 64) {
    return static_cast<uint32_t>((col >> 6) * (kKeyTile * 128)) + sw128_off(key, (col & 63) >> 3);
  } else {
    return static_cast<uint32_t>(key * (D * 2) + col * 2);
  }
}

template <int D>
__global__ void __launch_bounds__(256) sparse_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                                                          const __grid_constant__ CUtensorMap tmV,
                                                          const __nv_bfloat16* __restrict__ q,
                                                          const int32_t* __restrict__ pos, int n, int T, int Hq,
                                                          int Hkv, int G, int BR, float scale_log2,
                                                          __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                          int split_tiles, int max_splits, float* __restrict__ part_o,
                                                          float2* __restrict__ part_ml, unsigned int* status,
                                                          int check, int heads_fast) {
  using Cfg = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kAttnStages * 2 * Cfg::TILE_BYTES);
  uint64_t* empty = full + kAttnStages;

  const int nwarps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_blocks = (n + BR - 1) / BR;
  // grid (row block x split, KV head), or (KV head, row block x split) when heads_fast:
  // row blocks run heaviest first
  const int rbsp = static_cast<int>(heads_fast ? blockIdx.y : blockIdx.x);
  const int rb = n_blocks - 1 - rbsp / max_splits;
  const int sp = rbsp % max_splits;
  const int g = static_cast<int>(heads_fast ? blockIdx.x : blockIdx.y);
  const int row0 = rb * BR;
  const int row_end = min(n, row0 + BR);
  const int kmax = pos[row_end - 1];
  const int n_tiles_all = kmax / kKeyTile + 1;
  // key tiles [t_begin, n_tiles) of this split; a block whose keys fit in one split
  // writes its output directly, longer blocks write partial sums for the combine
  const int t_begin = sp * split_tiles;
  if (t_begin >= n_tiles_all) return;
  const int n_tiles = min(n_tiles_all, t_begin + split_tiles);
  const int n_split = min(max_splits, (n_tiles_all + split_tiles - 1) / split_tiles);

  const int hh = warp % G, rg = warp / G;
  const int h = g * G + hh;
  const int wrow0 = row0 + rg * 16;
  const int r_lo = wrow0 + (lane >> 2), r_hi = r_lo + 8;
  const int p_lo = r_lo < row_end ? pos[r_lo] : -1;
  const int p_hi = r_hi < row_end ? pos[r_hi] : -1;
  const int warp_kmax = wrow0 < row_end ? pos[min(row_end, wrow0 + 16) - 1] : -1;

  if (check && threadIdx.x == 0) {
    for (int r = row0; r < row_end; ++r) {
      const int p = pos[r];
      if (p < 0 || p >= T || (r > 0 && pos[r - 1] >= p)) {
        flag_status(status, QCF_DEV_BAD_INDEX);
        break;
      }
    }
  }

  // Q fragments (A operand of m16n8k16) straight from global memory.
  const int qc = (lane & 3) * 2;
  uint32_t qf[D / 16][4];
  {
    const size_t row_stride = static_cast<size_t>(Hq) * D;
    const __nv_bfloat16* qlo = q + static_cast<size_t>(r_lo) * row_stride + static_cast<size_t>(h) * D;
    const __nv_bfloat16* qhi = q + static_cast<size_t>(r_hi) * row_stride + static_cast<size_t>(h) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int k = ks * 16 + qc;
      qf[ks][0] = r_lo < row_end ? *reinterpret_cast<const uint32_t*>(qlo + k) : 0u;
      qf[ks][1] = r_hi < row_end ? *reinterpret_cast<const uint32_t*>(qhi + k) : 0u;
      qf[ks][2] = r_lo < row_end ? *reinterpret_cast<const uint32_t*>(qlo + k + 8) : 0u;
      qf[ks][3] = r_hi < row_end ? *reinterpret_cast<const uint32_t*>(qhi + k + 8) : 0u;
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nwarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  constexpr int boxes = D >= 64 ? D / 64 : 1;
  constexpr int box_cols = D >= 64 ? 64 : D;
  auto issue = [&](int t) {
    const int s = (t - t_begin) % kAttnStages;
    uint8_t* kb = smem + s * 2 * Cfg::TILE_BYTES;
    uint8_t* vb = kb + Cfg::TILE_BYTES;
    mbar_arrive_expect_tx(&full[s], 2 * Cfg::TILE_BYTES);
#pragma unroll
    for (int b = 0; b < boxes; ++b) {
      tma_load_2d(kb + b * kKeyTile * box_cols * 2, &tmK, &full[s], g * D + b * box_cols, t * kKeyTile);
      tma_load_2d(vb + b * kKeyTile * box_cols * 2, &tmV, &full[s], g * D + b * box_cols, t * kKeyTile);
    }
  };
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int t = t_begin; t < t_begin + kAttnStages && t < n_tiles; ++t) issue(t);
  }

  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

  bool ok = true;
  for (int t = t_begin; t < n_tiles; ++t) {
    const int s = (t - t_begin) % kAttnStages;
    const uint32_t par = ((t - t_begin) / kAttnStages) & 1;
    if (!mbar_wait(&full[s], par)) {
      flag_status(status, QCF_DEV_TIMEOUT);
      ok = false;
      break;
    }
    const int j0 = t * kKeyTile;
    if (j0 <= warp_kmax) {
      const uint32_t kaddr = smem_u32(smem + s * 2 * Cfg::TILE_BYTES);
      const uint32_t vaddr = kaddr + Cfg::TILE_BYTES;
      float sc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
      const int mi = lane >> 3, mr = lane & 7;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kaddr + tile_off<D>(np * 16 + (mi >> 1) * 8 + mr, ks * 16 + (mi & 1) * 8), b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * np], qf[ks], b0, b1);
          mma_bf16_16816(sc[2 * np + 1], qf[ks], b2, b3);
        }
      }
      // scale into log2 units, causal mask by true position, online softmax
      float tmax_lo = -INFINITY, tmax_hi = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = j0 + nt * 8 + qc + (e & 1);
          const int p = e < 2 ? p_lo : p_hi;
          const float x = key <= p ? sc[nt][e] * scale_log2 : -INFINITY;
          sc[nt][e] = x;
          if (e < 2) tmax_lo = fmaxf(tmax_lo, x); else tmax_hi = fmaxf(tmax_hi, x);
        }
      }
      tmax_lo = fmaxf(tmax_lo, __shfl_xor_sync(0xffffffffu, tmax_lo, 1));
      tmax_lo = fmaxf(tmax_lo, __shfl_xor_sync(0xffffffffu, tmax_lo, 2));
      tmax_hi = fmaxf(tmax_hi, __shfl_xor_sync(0xffffffffu, tmax_hi, 1));
      tmax_hi = fmaxf(tmax_hi, __shfl_xor_sync(0xffffffffu, tmax_hi, 2));
      const float mn_lo = fmaxf(m_lo, tmax_lo), mn_hi = fmaxf(m_hi, tmax_hi);
      const float base_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
      const float base_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
      const float alpha_lo = exp2f(m_lo - base_lo), alpha_hi = exp2f(m_hi - base_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      float rs_lo = 0.f, rs_hi = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - base_lo);
        sc[nt][1] = exp2f(sc[nt][1] - base_lo);
        sc[nt][2] = exp2f(sc[nt][2] - base_hi);
        sc[nt][3] = exp2f(sc[nt][3] - base_hi);
        rs_lo += sc[nt][0] + sc[nt][1];
        rs_hi += sc[nt][2] + sc[nt][3];
      }
      l_lo = l_lo * alpha_lo + rs_lo;
      l_hi = l_hi * alpha_hi + rs_hi;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        oacc[i][0] *= alpha_lo;
        oacc[i][1] *= alpha_lo;
        oacc[i][2] *= alpha_hi;
        oacc[i][3] *= alpha_hi;
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
        pa[1] = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
        pa[2] = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        pa[3] = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vaddr + tile_off<D>(kk * 16 + (mi & 1) * 8 + mr, dp * 16 + (mi >> 1) * 8), b0, b1, b2, b3);
          mma_bf16_16816(oacc[2 * dp], pa, b0, b1);
          mma_bf16_16816(oacc[2 * dp + 1], pa, b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (warp == 0) {
      if (lane == 0 && t + kAttnStages < n_tiles) {
        if (!mbar_wait(&empty[s], par)) {
          flag_status(status, QCF_DEV_TIMEOUT);
          ok = false;
        } else {
          issue(t + kAttnStages);
        }
      }
      __syncwarp();   // reconverge warp 0 before its next warp-wide MMA
    }
    if (!ok) break;
  }
  // On a timeout every warp gives up at its next wait (nothing more is issued);
  // the CTA then exits without writing.  No barrier follows, so warps that
  // finished normally cannot be stranded.
  if (!ok) return;

  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  if (n_split > 1) {   // unnormalised partial: O, running max (log2 units) and sum
    const size_t pstride = static_cast<size_t>(n) * Hq;
    if (r_lo < row_end) {
      float* po = part_o + (static_cast<size_t>(sp) * pstride + static_cast<size_t>(r_lo) * Hq + h) * D;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt)
        *reinterpret_cast<float2*>(po + dt * 8 + qc) = make_float2(oacc[dt][0], oacc[dt][1]);
      if ((lane & 3) == 0) part_ml[static_cast<size_t>(sp) * pstride + static_cast<size_t>(r_lo) * Hq + h] = make_float2(m_lo, l_lo);
    }
    if (r_hi < row_end) {
      float* po = part_o + (static_cast<size_t>(sp) * pstride + static_cast<size_t>(r_hi) * Hq + h) * D;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt)
        *reinterpret_cast<float2*>(po + dt * 8 + qc) = make_float2(oacc[dt][2], oacc[dt][3]);
      if ((lane & 3) == 0) part_ml[static_cast<size_t>(sp) * pstride + static_cast<size_t>(r_hi) * Hq + h] = make_float2(m_hi, l_hi);
    }
    return;
  }
  const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
  const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
  const size_t ostride = static_cast<size_t>(Hq) * D;
  if (r_lo < row_end) {
    __nv_bfloat16* op = o + static_cast<size_t>(r_lo) * ostride + static_cast<size_t>(h) * D;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt)
      *reinterpret_cast<uint32_t*>(op + dt * 8 + qc) = pack_bf16x2(oacc[dt][0] * inv_lo, oacc[dt][1] * inv_lo);
    if (lse && (lane & 3) == 0) lse[static_cast<size_t>(r_lo) * Hq + h] = (m_lo + log2f(l_lo)) * 0.69314718055994531f;
  }
  if (r_hi < row_end) {
    __nv_bfloat16* op = o + static_cast<size_t>(r_hi) * ostride + static_cast<size_t>(h) * D;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt)
      *reinterpret_cast<uint32_t*>(op + dt * 8 + qc) = pack_bf16x2(oacc[dt][2] * inv_hi, oacc[dt][3] * inv_hi);
    if (lse && (lane & 3) == 0) lse[static_cast<size_t>(r_hi) * Hq + h] = (m_hi + log2f(l_hi)) * 0.69314718055994531f;
  }
}

// ------------------------------------------------------------------ tensor-core (tcgen05) variant, D = 128
//
// One CTA = 128 score rows: BRp = floor(128 / G) consecutive recomputed rows x the
// G query heads of one KV head (row rho = p * G + hh), over key tiles of 128.  Seven warps:
//   warp 0     TMA producer for K: tiles of 128 keys (two 64-column boxes, 128B swizzle)
//              into a 3-stage ring; a stage is freed by the Q.K^T that read it
//   warp 1     TMEM allocation; one thread issues the tensor-core work in groups:
//              group g = { O += P_g V_g          (M=128, N=128, K=128 keys; P read from TMEM,
//                                                 V MN-major from shared memory),
//                          S_{g+2} = Q K_{g+2}^T  (M=128, N=128, K=128; Q read from TMEM) },
//              after S_0 and S_1.  Every dependency of group g lands on one mbarrier, so
//              the issuing thread reads one barrier per 16 MMAs of N=128: a barrier read
//              stalls the issuing thread longer than a small MMA takes, so long groups of
//              wide MMAs keep the tensor pipe fed.
//   warp 2     TMA producer for V: the same tiling, its own 3-stage ring, freed by P.V
//   warps 3-6  softmax, one score row per thread, 128 scores per tile: causal mask by
//              true position (boundary tiles only), online softmax in the exp2 domain with
//              the scale folded into one FFMA, P stored to TMEM as packed bf16 pairs, O
//              rescaled in TMEM only when a row max grows by more than 2^8.  S is double
//              buffered, so the scores of tile i+1 are ready while P.V of tile i runs.
// Group g's barrier go[g % 8] completes when: K_{g+2} has landed (or there is none), V_g
// has landed, and the four softmax warps have read S_g and written P_g.
// Q and P live in TMEM: each Q.K^T would otherwise re-read the Q slice from shared
// memory, whose bandwidth the operand reads and the TMA writes of K and V already share.
// TMEM columns: S_b at [128 b, 128 b + 128); O at [256, 384); Q at [384, 448) (128 bf16
// per row in 64 columns); P at [448, 512) (128 bf16 keys in 64 columns).
constexpr int kTcKeys = 128;
constexpr int kTcStages = 3;
constexpr int kTcGo = 8;                       // group barriers in flight
constexpr int kTcThreads = 224;
constexpr int kTcKVBytes = kTcKeys * 128 * 2;  // one K or V tile: 2 boxes of 128 keys x 64 columns
constexpr int kTcBoxBytes = kTcKeys * 128;     // one 64-column box
constexpr int kTcSmem = 2 * kTcStages * kTcKVBytes + 256 + 1024;
constexpr uint32_t kTcOCol = 256;              // first TMEM column of O
constexpr uint32_t kTcQCol = 384;              // first TMEM column of Q
constexpr uint32_t kTcPCol = 448;              // first TMEM column of P
constexpr uint32_t kTcGoCount = 10;            // K producer + V producer + 4 (S read) + 4 (P written)

__global__ void __launch_bounds__(kTcThreads, 1)
    sparse_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ pos, int n, int T, int Hq,
                          int Hkv, int G, int BRp, float scale_log2, __nv_bfloat16* __restrict__ o,
                          float* __restrict__ lse, int split_tiles, int max_splits, float* __restrict__ part_o,
                          float2* __restrict__ part_ml, unsigned int* status, int check, int heads_fast,
                          const int32_t* __restrict__ key0) {
  constexpr int D = 128;
  pdl_wait();  // q, pos and the cache come from the kernels before this one
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* kbuf = smem;  // stage st at st * KV
  uint8_t* vbuf = kbuf + kTcStages * kTcKVBytes;
  uint64_t* go = reinterpret_cast<uint64_t*>(vbuf + kTcStages * kTcKVBytes);
  uint64_t* k_init = go + kTcGo;  // K_0 and K_1, read by S_0 and S_1
  uint64_t* k_empty = k_init + 2;
  uint64_t* v_empty = k_empty + kTcStages;
  uint64_t* s_full = v_empty + kTcStages;  // [S buffer]
  uint64_t* pv_done = s_full + 2;
  uint64_t* q_ready = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_ready + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_blocks = (n + BRp - 1) / BRp;
  // grid (row block x split, KV head), or (KV head, row block x split) when heads_fast:
  // row blocks run heaviest first
  const int rbsp = static_cast<int>(heads_fast ? blockIdx.y : blockIdx.x);
  const int rb = n_blocks - 1 - rbsp / max_splits;
  const int sp = rbsp % max_splits;
  const int g = static_cast<int>(heads_fast ? blockIdx.x : blockIdx.y);
  const int row0 = rb * BRp;
  const int row_end = min(n, row0 + BRp);
  // the block's keys start at cache row kbase (several requests' caches in one buffer);
  // its positions count from there
  const int kbase = key0 ? key0[rb] : 0;
  const int n_tiles_all = (pos[row_end - 1] - kbase) / kTcKeys + 1;
  const int t_begin = sp * split_tiles;
  if (t_begin >= n_tiles_all) return;
  const int t_end = min(n_tiles_all, t_begin + split_tiles);
  const int n_split = min(max_splits, (n_tiles_all + split_tiles - 1) / split_tiles);
  const int nt = t_end - t_begin;  // >= 1

  if (threadIdx.x == 0) {
    for (int b = 0; b < kTcGo; ++b) mbar_init(&go[b], kTcGoCount);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&k_init[b], 1);
      mbar_init(&s_full[b], 1);
    }
    for (int st = 0; st < kTcStages; ++st) {
      mbar_init(&k_empty[st], 1);
      mbar_init(&v_empty[st], 1);
    }
    mbar_init(pv_done, 1);
    mbar_init(q_ready, 4);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 || warp == 2) {
    // ---- TMA producers: warp 0 streams K (tile t feeds group t - 2), warp 2 streams V (tile t feeds group t)
    if (lane == 0) {
      const bool is_k = warp == 0;
      const CUtensorMap* map = is_k ? &tmK : &tmV;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = is_k ? kbuf : vbuf;
      tma_prefetch_desc(map);
      bool ok = true;
      for (int i = 0; i < nt; ++i) {
        const int st = i % kTcStages;
        if (!mbar_wait(&empty[st], ((i / kTcStages) & 1) ^ 1u)) {
          flag_status(status, QCF_DEV_TIMEOUT);
          ok = false;
          break;
        }
        uint64_t* bar = is_k ? (i < 2 ? &k_init[i] : &go[(i - 2) % kTcGo]) : &go[i % kTcGo];
        mbar_arrive_expect_tx(bar, kTcKVBytes);
        uint8_t* dst = ring + st * kTcKVBytes;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
          tma_load_2d(dst + h2 * kTcBoxBytes, map, bar, g * D + h2 * 64, kbase + (t_begin + i) * kTcKeys);
      }
      // the last two groups have no K tile to wait for: their K share of the count arrives now
      if (is_k && ok)
        for (int gi = max(nt - 2, 0); gi < nt; ++gi) mbar_arrive(&go[gi % kTcGo]);
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTcKeys, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, true);
      auto issue_s = [&](int i) {  // S_{i % 2} = Q K_i^T, Q from TMEM
        const int st = i % kTcStages, b = i & 1;
        const uint32_t k_addr = smem_u32(kbuf + st * kTcKVBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_f16_ts(tmem_base + b * kTcKeys, tmem_base + kTcQCol + kk * 8,
                      sdesc_kmajor_sw128(k_addr + (kk >> 2) * kTcBoxBytes + (kk & 3) * 32), idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(&s_full[b]);
        umma_commit(&k_empty[st]);
      };
      bool ok = mbar_wait(q_ready, 0) && mbar_wait(&k_init[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        if (nt > 1) {
          ok = mbar_wait(&k_init[1], 0);
          tc_fence_after();
          if (ok) issue_s(1);
        }
      }
      for (int gi = 0; gi < nt && ok; ++gi) {
        if (!mbar_wait(&go[gi % kTcGo], (gi / kTcGo) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // O += P_gi V_gi first: the single P buffer is free again as soon as it completes,
        // while S_{gi+2} is needed only after the softmax of tile gi+1
        const int st = gi % kTcStages;
        const uint32_t v_addr = smem_u32(vbuf + st * kTcKVBytes);
#pragma unroll
        for (int kk = 0; kk < kTcKeys / 16; ++kk)
          umma_f16_ts(tmem_base + kTcOCol, tmem_base + kTcPCol + kk * 8,
                      sdesc_mnmajor_sw128(v_addr + kk * 2048, kTcBoxBytes), idesc_o, (gi > 0 || kk > 0) ? 1u : 0u);
        umma_commit(pv_done);
        umma_commit(&v_empty[st]);
        if (gi + 2 < nt) issue_s(gi + 2);
      }
      if (!ok) flag_status(status, QCF_DEV_TIMEOUT);
    }
  } else {
    // ---- softmax: thread = score row
    constexpr unsigned kAll = 0xffffffffu;
    const int quarter = warp & 3;
    const int rho = quarter * 32 + lane;
    const int p_local = rho / G, hh = rho - p_local * G;
    const int r = row0 + p_local;
    const bool valid = p_local < BRp && r < row_end;
    const int prow = valid ? pos[r] - kbase : -1;   // relative to the block's first key
    const int h = g * G + hh;
    // positions ascend over all rows, or within each block when blocks have their own key base
    if (check && valid && (prow < 0 || prow + kbase >= T || (r > (key0 ? row0 : 0) && pos[r - 1] - kbase >= prow)))
      flag_status(status, QCF_DEV_BAD_INDEX);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    {  // the Q row into TMEM as 64 packed bf16 pairs (all 16 loads in flight before the stores)
      const uint4* src = reinterpret_cast<const uint4*>(q + (static_cast<size_t>(valid ? r : 0) * Hq + h) * D);
      uint32_t w[64];
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const uint4 v = valid ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
        w[4 * ch] = v.x;
        w[4 * ch + 1] = v.y;
        w[4 * ch + 2] = v.z;
        w[4 * ch + 3] = v.w;
      }
      tmem_st32u(tmem_base + lane_base + kTcQCol, w);
      tmem_st32u(tmem_base + lane_base + kTcQCol + 32, w + 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    const uint32_t o_tm = tmem_base + lane_base + kTcOCol;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < nt; ++i) {
      uint64_t* gob = &go[i % kTcGo];
      const int b = i & 1;
      if (!__all_sync(kAll, mbar_wait(&s_full[b], (i >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[kTcKeys];
      tmem_ld64(tmem_base + lane_base + b * kTcKeys, sv);
      tmem_ld64(tmem_base + lane_base + b * kTcKeys + 64, sv + 64);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(gob);  // S_i read: its buffer may take S_{i+2}
      const int j0 = (t_begin + i) * kTcKeys;
      if (j0 + kTcKeys - 1 > prow) {
#pragma unroll
        for (int j = 0; j < kTcKeys; ++j)
          if (j0 + j > prow) sv[j] = -INFINITY;
      }
      float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
      for (int j = 4; j < kTcKeys; j += 4) {
        mx0 = fmaxf(mx0, sv[j]);
        mx1 = fmaxf(mx1, sv[j + 1]);
        mx2 = fmaxf(mx2, sv[j + 2]);
        mx3 = fmaxf(mx3, sv[j + 3]);
      }
      const float tmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale_log2;
      // rescale lazily: keep the old max unless a row's max grew by more than 2^8
      const bool grow = tmax > m + 8.0f;
      if (__any_sync(kAll, grow)) {
        const float m_new = grow ? tmax : m;
        if (i > 0) {  // O holds the tiles so far: wait for the last P.V, then scale
          if (!__all_sync(kAll, mbar_wait(pv_done, (i - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = (m == -INFINITY) ? 0.f : fast_exp2(m - m_new);
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float ov[32];
            tmem_ld32(o_tm + c * 32, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] *= f;
            tmem_st32(o_tm + c * 32, ov);
          }
          l *= f;
        }
        m = m_new;
      }
      const float nm = (m == -INFINITY) ? 0.f : -m;  // m = -inf only when every key so far is masked
      float rs0 = 0.f, rs1 = 0.f, rs2 = 0.f, rs3 = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        const float p0 = fast_exp2(fmaf(sv[2 * e], scale_log2, nm));
        const float p1 = fast_exp2(fmaf(sv[2 * e + 1], scale_log2, nm));
        const float p2 = fast_exp2(fmaf(sv[2 * e + 2], scale_log2, nm));
        const float p3 = fast_exp2(fmaf(sv[2 * e + 3], scale_log2, nm));
        rs0 += p0;
        rs1 += p1;
        rs2 += p2;
        rs3 += p3;
        pk[e] = pack_bf16x2(p0, p1);  // key 2e in the low half
        pk[e + 1] = pack_bf16x2(p2, p3);
      }
      l += (rs0 + rs1) + (rs2 + rs3);
      // the P buffer was last read by the previous tile's P.V
      if (i > 0 && !__all_sync(kAll, mbar_wait(pv_done, (i - 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st32u(tmem_base + lane_base + kTcPCol, pk);
      tmem_st32u(tmem_base + lane_base + kTcPCol + 32, pk + 32);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(gob);  // P_i written
    }
    if (ok && !__all_sync(kAll, mbar_wait(pv_done, (nt - 1) & 1))) ok = false;
    if (!ok) {
      flag_status(status, QCF_DEV_TIMEOUT);
    } else {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t pstride = static_cast<size_t>(n) * Hq;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tmem_ld32(o_tm + c * 32, ov);
        if (!valid) continue;
        if (n_split > 1) {
          float* po = part_o + (static_cast<size_t>(sp) * pstride + static_cast<size_t>(r) * Hq + h) * D + c * 32;
#pragma unroll
          for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4*>(po + e) = make_float4(ov[e], ov[e + 1], ov[e + 2], ov[e + 3]);
        } else {
          __nv_bfloat16* op = o + (static_cast<size_t>(r) * Hq + h) * D + c * 32;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 u;
            u.x = pack_bf16x2(ov[e] * inv, ov[e + 1] * inv);
            u.y = pack_bf16x2(ov[e + 2] * inv, ov[e + 3] * inv);
            u.z = pack_bf16x2(ov[e + 4] * inv, ov[e + 5] * inv);
            u.w = pack_bf16x2(ov[e + 6] * inv, ov[e + 7] * inv);
            *reinterpret_cast<uint4*>(op + e) = u;
          }
        }
      }
      if (valid) {
        if (n_split > 1)
          part_ml[static_cast<size_t>(sp) * pstride + static_cast<size_t>(r) * Hq + h] = make_float2(m, l);
        else if (lse)
          lse[static_cast<size_t>(r) * Hq + h] = (m + log2f(l)) * 0.69314718055994531f;
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

// Merges the key-range partials of rows whose block was split: one warp per
// (row, head), splits summed in order (deterministic).
template <int D>
__global__ void attn_combine_kernel(const int32_t* __restrict__ pos, int n, int Hq, int BR, int tile, int split_tiles,
                                    int max_splits, const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                                    __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  pdl_wait();
  pdl_launch_dependents();
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= n * Hq) return;
  const int row = w / Hq, h = w - row * Hq;
  const int rb = row / BR;
  const int row_end = min(n, rb * BR + BR);
  const int n_tiles_all = pos[row_end - 1] / tile + 1;
  const int n_split = min(max_splits, (n_tiles_all + split_tiles - 1) / split_tiles);
  if (n_split <= 1) return;
  const size_t pstride = static_cast<size_t>(n) * Hq;
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, part_ml[s * pstride + static_cast<size_t>(row) * Hq + h].x);
  constexpr int PER = (D + 31) / 32;   // elements d = lane + 32 i, d < D
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float L = 0.f;
  for (int s = 0; s < n_split; ++s) {
    const float2 ml = part_ml[s * pstride + static_cast<size_t>(row) * Hq + h];
    if (!(ml.y > 0.f)) continue;
    const float f = exp2f(ml.x - M);
    L += ml.y * f;
    const float* po = part_o + (s * pstride + static_cast<size_t>(row) * Hq + h) * D;
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (lane + 32 * i < D) acc[i] += po[lane + 32 * i] * f;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* op = o + (static_cast<size_t>(row) * Hq + h) * D;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (lane + 32 * i < D) op[lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
  if (lse && lane == 0) lse[static_cast<size_t>(row) * Hq + h] = (M + log2f(L)) * 0.69314718055994531f;
}

struct AttnPlan {
  int G, BR, tile, n_blocks, split_tiles, max_splits;   // tile: keys per pipeline step
};

// Long row blocks are split over key ranges only when the grid is too small to
// balance by itself (the fused path: few rows, the query block sees every key).
static AttnPlan plan_attn(int n, int T, int Hq, int Hkv, int D) {
  AttnPlan p;
  p.G = Hq / Hkv;
  // rows per CTA: the tensor-core kernel (D = 128) fills 128 score rows, the warp-MMA kernel 16 per warp
  p.BR = D == 128 ? 128 / p.G : 16 * (p.G >= 8 ? 1 : 8 / p.G);
  p.n_blocks = (n + p.BR - 1) / p.BR;
  p.tile = D == 128 ? kTcKeys : kKeyTile;
  const int max_tiles = (T + p.tile - 1) / p.tile;
  p.split_tiles = max_tiles;
  p.max_splits = 1;
  const int ctas = p.n_blocks * Hkv, sms = num_sms();
  if (D == 128) {
    // tensor-core kernel, one CTA per SM: a CTA's set-up and drain cost more than the
    // imbalance of unsplit rows once every SM has a CTA (8B recompute shape: 81 us
    // unsplit vs 99 us with 4 splits plus the combine), so split only a grid smaller
    // than the SM count, into at most 4 ranges of at least 8 tiles of 128 keys
    if (ctas < sms && max_tiles > 8) {
      p.max_splits = std::min(4, (sms + ctas - 1) / ctas);
      p.split_tiles = std::max(8, (max_tiles + p.max_splits - 1) / p.max_splits);
      p.max_splits = (max_tiles + p.split_tiles - 1) / p.split_tiles;
    }
  } else if (ctas < 4 * sms && max_tiles > 16) {
    p.max_splits = 4;
    p.split_tiles = (max_tiles + p.max_splits - 1) / p.max_splits;
    if (p.split_tiles < 8) p.split_tiles = 8;
    p.max_splits = (max_tiles + p.split_tiles - 1) / p.split_tiles;
  }
  return p;
}

size_t attn_workspace_size(int n, int T, int Hq, int Hkv, int D) {
  if (n <= 0 || T <= 0 || Hkv <= 0 || Hq % Hkv) return 0;
  const AttnPlan p = plan_attn(n, T, Hq, Hkv, D);
  if (p.max_splits <= 1) return 0;
  return align_up(static_cast<size_t>(p.max_splits) * n * Hq * D * sizeof(float), 256) +
         align_up(static_cast<size_t>(p.max_splits) * n * Hq * sizeof(float2), 256);
}

template <int D>
static qcf_status attn_launch_d(const __nv_bfloat16* q, const int32_t* pos, int n, const __nv_bfloat16* K,
                                const __nv_bfloat16* V, int T, int Hq, int Hkv, float scale, __nv_bfloat16* o,
                                float* lse, void* ws, size_t ws_bytes, cudaStream_t st, KernelClass kc, bool pdl,
                                const int32_t* key0) {
  using Cfg = AttnCfg<D>;
  AttnPlan plan = plan_attn(n, T, Hq, Hkv, D);
  if (key0) {  // blocks with their own key base: whole key ranges only (the combine reads positions from 0)
    plan.split_tiles = (T + plan.tile - 1) / plan.tile;
    plan.max_splits = 1;
  }
  const int G = plan.G;
  const int BR = plan.BR;
  const int warps = G * (BR / 16);
  float* part_o = nullptr;
  float2* part_ml = nullptr;
  if (plan.max_splits > 1) {
    const size_t ob = align_up(static_cast<size_t>(plan.max_splits) * n * Hq * D * sizeof(float), 256);
    if (!ws || ws_bytes < attn_workspace_size(n, T, Hq, Hkv, D))
      return set_error(QCF_ERR_WORKSPACE, "sparse_causal_attn: workspace %zu < %zu", ws_bytes,
                       attn_workspace_size(n, T, Hq, Hkv, D));
    part_o = static_cast<float*>(ws);
    part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + ob);
  }
  CUtensorMap tk, tv;
  const uint64_t width = static_cast<uint64_t>(Hkv) * D;
  const uint32_t box_cols = D >= 64 ? 64 : D;
  const CUtensorMapSwizzle sw = Cfg::SW128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (!encode_tmap_2d(&tk, K, width, T, width * 2, box_cols, plan.tile, sw) ||
      !encode_tmap_2d(&tv, V, width, T, width * 2, box_cols, plan.tile, sw))
    return set_error(QCF_ERR_CUDA, "sparse_causal_attn: tensor map encoding failed");
  static PerDevice<cudaError_t> smem_attr;
  const cudaError_t attr = smem_attr.get(current_device(), [] {
    return cudaFuncSetAttribute(sparse_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  });
  if (attr != cudaSuccess) return cuda_error(attr, "sparse_causal_attn: smem attribute");
  // When every head's K and V fit in L2 together (the fused prefill's layers), the
  // KV heads go fastest in launch order so each head's heaviest row blocks start in
  // the first wave; larger caches keep head-major order, whose concurrent CTAs share
  // one head's K/V stream in L2.
  const int rbs = plan.n_blocks * plan.max_splits;
  const int heads_fast =
      static_cast<size_t>(T) * Hkv * D * 2 * 2 <= (static_cast<size_t>(64) << 20) && rbs <= 65535 ? 1 : 0;
  dim3 grid = heads_fast ? dim3(Hkv, rbs) : dim3(rbs, Hkv);
  const float scale_log2 = scale * 1.4426950408889634f;
  if constexpr (D == 128) {
    static PerDevice<cudaError_t> smem_attr_tc;
    const cudaError_t attr_tc = smem_attr_tc.get(current_device(), [] {
      return cudaFuncSetAttribute(sparse_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    });
    if (attr_tc != cudaSuccess) return cuda_error(attr_tc, "sparse_causal_attn: smem attribute");
    LaunchScope ls(kc, st);
    if (pdl) {
      cudaError_t e = launch_pdl(sparse_attn_tc_kernel, grid, dim3(kTcThreads), kTcSmem, st, tk, tv, q, pos, n, T, Hq,
                                 Hkv, G, BR, scale_log2, o, lse, plan.split_tiles, plan.max_splits, part_o, part_ml,
                                 device_status_ptr(), check_enabled() ? 1 : 0, heads_fast, key0);
      if (e != cudaSuccess) return cuda_error(e, "sparse_causal_attn: launch");
    } else {
      sparse_attn_tc_kernel<<<grid, kTcThreads, kTcSmem, st>>>(tk, tv, q, pos, n, T, Hq, Hkv, G, BR, scale_log2, o, lse,
                                                                plan.split_tiles, plan.max_splits, part_o, part_ml,
                                                                device_status_ptr(), check_enabled() ? 1 : 0, heads_fast,
                                                                key0);
    }
  } else {
    LaunchScope ls(kc, st);
    sparse_attn_kernel<D><<<grid, warps * 32, Cfg::SMEM_BYTES, st>>>(
        tk, tv, q, pos, n, T, Hq, Hkv, G, BR, scale_log2, o, lse, plan.split_tiles, plan.max_splits, part_o, part_ml,
        device_status_ptr(), check_enabled() ? 1 : 0, heads_fast);
  }
  if (plan.max_splits > 1) {
    LaunchScope ls(kc == KC_ATTN ? KC_ATTN_COMBINE : kc, st);
    const int warps_total = n * Hq;
    if (pdl) {
      cudaError_t e = launch_pdl(attn_combine_kernel<D>, dim3((warps_total + 7) / 8), dim3(256), 0, st, pos, n, Hq, BR,
                                 plan.tile, plan.split_tiles, plan.max_splits, part_o, part_ml, o, lse);
      if (e != cudaSuccess) return cuda_error(e, "sparse_causal_attn: combine launch");
    } else {
      attn_combine_kernel<D><<<(warps_total + 7) / 8, 256, 0, st>>>(pos, n, Hq, BR, plan.tile, plan.split_tiles,
                                                                    plan.max_splits, part_o, part_ml, o, lse);
    }
  }
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "sparse_causal_attn: launch");
}

qcf_status attn_launch(const __nv_bfloat16* q, const int32_t* pos, int n, const __nv_bfloat16* K, const __nv_bfloat16* V,
                       int T, int Hq, int Hkv, int D, float scale, __nv_bfloat16* o, float* lse, void* ws,
                       size_t ws_bytes, cudaStream_t st, KernelClass kc, bool pdl, const int32_t* key0) {
  if (n <= 0) return QCF_OK;
  if (key0 && D != 128) return set_error(QCF_ERR_UNSUPPORTED, "sparse_causal_attn: per-block key bases need D = 128");
  switch (D) {  // the warp-MMA kernel (D = 16, 64) is launched plainly; its combine may still be programmatic
    case 16: return attn_launch_d<16>(q, pos, n, K, V, T, Hq, Hkv, scale, o, lse, ws, ws_bytes, st, kc, pdl, nullptr);
    case 64: return attn_launch_d<64>(q, pos, n, K, V, T, Hq, Hkv, scale, o, lse, ws, ws_bytes, st, kc, pdl, nullptr);
    case 128: return attn_launch_d<128>(q, pos, n, K, V, T, Hq, Hkv, scale, o, lse, ws, ws_bytes, st, kc, pdl, key0);
    default: return set_error(QCF_ERR_SHAPE, "sparse_causal_attn: head dim %d unsupported", D);
  }
}

}  // namespace qcf

using namespace qcf;

extern "C" {

size_t qcf_sparse_causal_attn_workspace_size(int n, int T, int Hq, int Hkv, int D) {
  return attn_workspace_size(n, T, Hq, Hkv, D);
}

qcf_status qcf_sparse_causal_attn(const qcf_bf16* q, const int32_t* pos, int n, const qcf_bf16* K, const qcf_bf16* V,
                                  int T, int Hq, int Hkv, int D, float scale, qcf_bf16* o, float* lse, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (!q || !pos || !K || !V || !o) return set_error(QCF_ERR_INVALID_ARG, "qcf_sparse_causal_attn: NULL pointer");
  if (n < 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Hq / Hkv > 8 || (D != 16 && D != 64 && D != 128))
    return set_error(QCF_ERR_SHAPE, "qcf_sparse_causal_attn: n=%d T=%d Hq=%d Hkv=%d D=%d", n, T, Hq, Hkv, D);
  if (take_fault(4) || !aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(o))
    return set_error(QCF_ERR_ALIGN, "qcf_sparse_causal_attn: pointers must be 16-byte aligned");
  if (take_fault(1)) return set_error(QCF_ERR_INVALID_ARG, "qcf_sparse_causal_attn: injected invalid index table");
  if (ws_bytes < qcf_sparse_causal_attn_workspace_size(n, T, Hq, Hkv, D))
    return set_error(QCF_ERR_WORKSPACE, "qcf_sparse_causal_attn: workspace too small");
  return attn_launch(reinterpret_cast<const __nv_bfloat16*>(q), pos, n, reinterpret_cast<const __nv_bfloat16*>(K),
                     reinterpret_cast<const __nv_bfloat16*>(V), T, Hq, Hkv, D, scale,
                     reinterpret_cast<__nv_bfloat16*>(o), lse, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
