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
constexpr int kPtBoxBytes = kPtKeys * 128;            // 128 keys x 64 bf16
constexpr int kPtTileBytes = 2 * kPtBoxBytes;         // 128 keys x 128 bf16
constexpr int kPtQBytes = 4 * 128 * 128;              // 2 row tiles x 2 column boxes x 128 rows x 64 bf16
constexpr int kPtThreads = 576;                       // producer, MMA, 16 softmax warps
// pass 1 keeps the query rows in tensor memory and gives shared memory to a deeper K ring;
// pass 2 needs them in shared memory (they are the B operand of K Q^T)
template <bool PASS2>
struct PtCfg {
  static constexpr int kStages = PASS2 ? 4 : 6;
  static constexpr int kQBytes = PASS2 ? kPtQBytes : 0;
  static constexpr int kSmem = kQBytes + kStages * kPtTileBytes + 6144 + 1024;
};

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
    profile_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                      const __nv_bfloat16* __restrict__ q, int nq, int Hq, int C, int G, int R, int RT, int n_rt,
                      int n_rg, int tpc, int n_kc, float scale_log2, float2* __restrict__ stats,
                      float* __restrict__ part, unsigned int* __restrict__ counters, float* __restrict__ scores,
                      unsigned int* status) {
  using Cfg = PtCfg<PASS2>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* qbuf = smem;                      // pass 2: box (column half hb, row tile t) at hb * 32 KB + t * 16 KB
  uint8_t* kbuf = smem + Cfg::kQBytes;       // stage st at st * 32 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(kbuf + S * kPtTileBytes);
  uint64_t* q_full = bars;                   // pass 1: the query rows are in tensor memory
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + S;
  uint64_t* s_full = k_empty + S;            // pass 1: per row tile; pass 2: per accumulator buffer
  uint64_t* s_free = s_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_free + 2);
  uint32_t* last_flag = tmem_slot + 1;
  float* mp = reinterpret_cast<float*>(kbuf + S * kPtTileBytes + 1024);   // [2][128] M' (pass 2)
  float* red = mp + 256;                                                  // [2][4][128] (or [2][256] float2)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kc = blockIdx.x, g = blockIdx.y, rg = blockIdx.z;
  const int n_part = gridDim.y * n_rg;
  const int n_tiles = (C + kPtKeys - 1) / kPtKeys;
  const int t0 = kc * tpc;
  const int t1 = min(n_tiles, t0 + tpc);
  const int nt = t1 - t0;  // >= 1 by the plan
  const int n_rt_cta = min(2, n_rt - rg * 2);
  // TMEM columns.  Pass 1: S of row tile t at t * 128 (one buffer per row tile: the two row
  // tiles' MMAs alternate, so one tile's accumulator is read while the other's is computed),
  // the query rows (128 bf16 as 64 packed columns) at 256 + t * 64.  Pass 2: S^T of tile i
  // at (i & 1) * 256, 128 columns per row tile.
  constexpr uint32_t kQCol = 256;

  if (!PASS2) {
    pdl_launch_dependents();  // pass 2 may start its set-up and its key stream as SMs free up
    if (kc == 0 && g == 0 && rg == 0)
      for (int i = threadIdx.x; i < n_kc; i += blockDim.x) counters[i] = 0u;
  }
  if (threadIdx.x == 0) {
    mbar_init(q_full, PASS2 ? 1 : 8 * n_rt_cta);
    for (int st = 0; st < S; ++st) {
      mbar_init(&k_full[st], 1);
      mbar_init(&k_empty[st], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], PASS2 ? 8 * n_rt_cta : 8);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (PASS2 && RT < 128) {
    // rows RT..127 of each query row tile lie outside the TMA boxes: zero them, so the
    // transposed scores hold zeros (not stale bits) in those columns
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
    // ---- TMA producer: (pass 2) the CTA's query rows once, then the chunk's K tiles
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      if (PASS2) {
        tma_prefetch_desc(&tmQ);
        mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(n_rt_cta * 2 * RT * 128));
        for (int t = 0; t < n_rt_cta; ++t)
#pragma unroll
          for (int hb = 0; hb < 2; ++hb)
            tma_load_3d(qbuf + hb * 32768 + t * 16384, &tmQ, q_full, hb * 64, g * G, (rg * 2 + t) * R);
      }
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int st = i % S;
        if (!mbar_wait(&k_empty[st], ((i / S) & 1) ^ 1u)) {
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
      for (int i = max(0, issued - S); i < issued; ++i)
        if (!mbar_wait(&k_full[i % S], (i / S) & 1)) flag_status(status, QCF_DEV_TIMEOUT);
      if (PASS2 && !mbar_wait(q_full, 0)) flag_status(status, QCF_DEV_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint32_t k_addr = smem_u32(kbuf);
      bool ok = mbar_wait(q_full, 0);
      int done = 0;
      for (int i = 0; i < nt && ok; ++i) {
        const int st = i % S;
        if (!mbar_wait(&k_full[st], (i / S) & 1)) {
          ok = false;
          break;
        }
        const uint32_t kst = k_addr + st * kPtTileBytes;
        if (!PASS2) {
          // S_t = Q_t K^T, Q_t read from tensor memory, one accumulator per row tile
          constexpr uint32_t idesc_s = idesc_bf16_f32(128, kPtKeys);
          for (int t = 0; t < n_rt_cta && ok; ++t) {
            if (!mbar_wait(&s_free[t], (i & 1) ^ 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_f16_ts(tmem_base + t * 128, tmem_base + kQCol + t * 64 + kk * 8,
                          sdesc_kmajor_sw128(kst + (kk >> 2) * kPtBoxBytes + (kk & 3) * 32), idesc_s, kk > 0 ? 1u : 0u);
            umma_commit(&s_full[t]);
          }
          if (!ok) break;
        } else {
          // S^T = K Q^T into the buffer of this tile's parity
          const int b = i & 1;
          if (!mbar_wait(&s_free[b], ((i >> 1) & 1) ^ 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t q_addr = smem_u32(qbuf);
          const uint32_t idesc_t = idesc_bf16_f32(128, 128 * n_rt_cta);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_f16(tmem_base + b * 256, sdesc_kmajor_sw128(kst + (kk >> 2) * kPtBoxBytes + (kk & 3) * 32),
                     sdesc_kmajor_sw128(q_addr + (kk >> 2) * 32768 + (kk & 3) * 32), idesc_t, kk > 0 ? 1u : 0u);
          umma_commit(&s_full[b]);
        }
        umma_commit(&k_empty[st]);
        done = i + 1;
      }
      if (!ok) flag_status(status, QCF_DEV_TIMEOUT);
      // the last tile's MMAs and their barrier arrivals are complete before tensor memory
      // is freed and the CTA's shared memory is released
      if (done > 0 && !mbar_wait(&k_empty[(done - 1) % S], ((done - 1) / S) & 1)) flag_status(status, QCF_DEV_TIMEOUT);
    }
  } else {
    // ---- softmax warps, four warpgroups: warpgroup wg serves row tile t = wg & 1 and half
    // ch = wg >> 1 of the tile's 128 accumulator columns (keys in pass 1, score rows in
    // pass 2); a warp reaches the TMEM lanes of quarter warp % 4
    constexpr unsigned kAll = 0xffffffffu;
    const int wg = (warp - 2) >> 2;
    const int t = wg & 1, ch = wg >> 1;
    const int quarter = warp & 3;
    const int l128 = quarter * 32 + lane;
    const int sm_tid = threadIdx.x - 64;  // 0..511 over the softmax warps
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const bool active = t < n_rt_cta;
    const size_t part_row = static_cast<size_t>(g * n_rg + rg);
    const uint32_t acc_col = static_cast<uint32_t>(t * 128 + ch * 64);
    if (!PASS2) {
      // this thread's half of its score row's query vector into tensor memory (rows past the
      // query or in the padding of a row tile are zeros)
      if (active) {
        const int r = (rg * 2 + t) * R + l128 / G;
        const bool valid = l128 < RT && r < nq;
        const uint4* src = reinterpret_cast<const uint4*>(
            q + (static_cast<size_t>(valid ? r : 0) * Hq + g * G + (valid ? l128 % G : 0)) * 128 + ch * 64);
        uint32_t w[32];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const uint4 v = valid ? src[c8] : make_uint4(0u, 0u, 0u, 0u);
          w[4 * c8] = v.x;
          w[4 * c8 + 1] = v.y;
          w[4 * c8 + 2] = v.z;
          w[4 * c8 + 3] = v.w;
        }
        tmem_st32u(tmem_base + lane_base + kQCol + t * 64 + ch * 32, w);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
      }
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < nt && active; ++i) {
        if (!__all_sync(kAll, mbar_wait(&s_full[t], i & 1))) {
          flag_status(status, QCF_DEV_TIMEOUT);
          break;
        }
        tc_fence_after();
        float v[64];
        tmem_ld64(tmem_base + lane_base + t * 128 + ch * 64, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[t]);
        const int j0 = (t0 + i) * kPtKeys + ch * 64;
        if (j0 + 64 > C) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (j0 + k >= C) v[k] = -INFINITY;
        }
        float a0 = v[0], a1 = v[1], a2 = v[2], a3 = v[3];
#pragma unroll
        for (int k = 4; k < 64; k += 4) {
          a0 = fmaxf(a0, v[k]);
          a1 = fmaxf(a1, v[k + 1]);
          a2 = fmaxf(a2, v[k + 2]);
          a3 = fmaxf(a3, v[k + 3]);
        }
        const float mn = fmaxf(m, fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * scale_log2);
        const float base = mn == -INFINITY ? 0.f : mn;
        const float nb = -base;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f, s5 = 0.f, s6 = 0.f, s7 = 0.f;
#pragma unroll
        for (int k = 0; k < 64; k += 8) {
          s0 += fast_exp2(fmaf(v[k], scale_log2, nb));
          s1 += fast_exp2(fmaf(v[k + 1], scale_log2, nb));
          s2 += fast_exp2(fmaf(v[k + 2], scale_log2, nb));
          s3 += fast_exp2(fmaf(v[k + 3], scale_log2, nb));
          s4 += fast_exp2(fmaf(v[k + 4], scale_log2, nb));
          s5 += fast_exp2(fmaf(v[k + 5], scale_log2, nb));
          s6 += fast_exp2(fmaf(v[k + 6], scale_log2, nb));
          s7 += fast_exp2(fmaf(v[k + 7], scale_log2, nb));
        }
        l = l * fast_exp2(m - base) + (((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)));
        m = mn;
      }
      // the two column halves of a row merge their statistics
      float2* half_stats = reinterpret_cast<float2*>(red);  // [2 row tiles][128]
      if (ch == 1 && active) half_stats[t * 128 + l128] = make_float2(m, l);
      asm volatile("bar.sync 1, 512;" ::: "memory");
      if (ch == 0 && active) {
        const float2 o = half_stats[t * 128 + l128];
        const float mn = fmaxf(m, o.x);
        const float base = mn == -INFINITY ? 0.f : mn;
        const float lt = l * fast_exp2(m - base) + o.y * fast_exp2(o.x - base);
        stats[(part_row * n_kc + kc) * 256 + t * 128 + l128] = make_float2(mn, lt);
      }
    } else {
      pdl_wait();  // the statistics of pass 1
      // M' = M + log2(L) of each score row from the chunks' partial statistics: two threads
      // per row, each merging half of the chunks with four loads in flight, then the halves
      // meet in shared memory.  Rows past the query or in the padding of a row tile get
      // +inf, which zeroes their terms.
      {
        const int row = sm_tid & 255, half = sm_tid >> 8;
        const int per = (n_kc + 1) >> 1;
        const int k_lo = half * per, k_hi = min(n_kc, k_lo + per);
        const float2* sp = stats + part_row * n_kc * 256 + row;
        float M = -INFINITY, L = 0.f;
        auto merge = [&](float2 sv) {
          const float mn = fmaxf(M, sv.x);
          const float base = mn == -INFINITY ? 0.f : mn;
          L = L * exp2f(M - base) + sv.y * exp2f(sv.x - base);
          M = mn;
        };
        int k = k_lo;
        for (; k + 4 <= k_hi; k += 4) {
          const float2 a0 = sp[static_cast<size_t>(k) * 256], a1 = sp[static_cast<size_t>(k + 1) * 256];
          const float2 a2 = sp[static_cast<size_t>(k + 2) * 256], a3 = sp[static_cast<size_t>(k + 3) * 256];
          merge(a0);
          merge(a1);
          merge(a2);
          merge(a3);
        }
        for (; k < k_hi; ++k) merge(sp[static_cast<size_t>(k) * 256]);
        float2* halves = reinterpret_cast<float2*>(red);  // [2][256]
        halves[half * 256 + row] = make_float2(M, L);
        asm volatile("bar.sync 1, 512;" ::: "memory");
        if (sm_tid < 256) {
          const float2 o = halves[256 + row];
          merge(o);
          const int tt = row >> 7, rr = row & 127;
          const int r = (rg * 2 + tt) * R + rr / G;
          mp[row] = (tt < n_rt_cta && rr < RT && r < nq && L > 0.f) ? M + log2f(L) : INFINITY;
        }
      }
      asm volatile("bar.sync 1, 512;" ::: "memory");
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
            float v[64];
            tmem_ld64(tmem_base + lane_base + b * 256 + acc_col, v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[b]);
            const float4* m4 = reinterpret_cast<const float4*>(mp + acc_col);
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f, s5 = 0.f, s6 = 0.f, s7 = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
              const float4 ma = m4[k], mb = m4[k + 1];
              s0 += fast_exp2(fmaf(v[4 * k], scale_log2, -ma.x));
              s1 += fast_exp2(fmaf(v[4 * k + 1], scale_log2, -ma.y));
              s2 += fast_exp2(fmaf(v[4 * k + 2], scale_log2, -ma.z));
              s3 += fast_exp2(fmaf(v[4 * k + 3], scale_log2, -ma.w));
              s4 += fast_exp2(fmaf(v[4 * k + 4], scale_log2, -mb.x));
              s5 += fast_exp2(fmaf(v[4 * k + 5], scale_log2, -mb.y));
              s6 += fast_exp2(fmaf(v[4 * k + 6], scale_log2, -mb.z));
              s7 += fast_exp2(fmaf(v[4 * k + 7], scale_log2, -mb.w));
            }
            acc = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
          }
        }
        // the four partial sums of a key meet in shared memory; the barrier also lets a
        // timed-out warp leave the loop together with every other softmax warp
        red[(i & 1) * 512 + wg * 128 + l128] = acc;
        if (bar_red_or(1, 512, !ok)) break;
        const int j = tk * kPtKeys + sm_tid;
        if (sm_tid < 128 && j < C) {
          const float* rp = red + (i & 1) * 512 + sm_tid;
          part[part_row * C + j] = (rp[0] + rp[256]) + (rp[128] + rp[384]);
        }
      }
      // the last of the chunk's CTAs to finish adds the n_part partial vectors in order
      __threadfence();
      asm volatile("bar.sync 1, 512;" ::: "memory");
      if (sm_tid == 0) {
        const unsigned int prev = atomicAdd(&counters[kc], 1u);
        *last_flag = prev == static_cast<unsigned int>(n_part - 1) ? 1u : 0u;
      }
      asm volatile("bar.sync 1, 512;" ::: "memory");
      if (*last_flag) {
        __threadfence();
        // four keys per thread at a time, every load of a round independent of the sums
        const int j_end = min(C, t1 * kPtKeys);
        for (int j = t0 * kPtKeys + sm_tid; j < j_end; j += 4 * 512) {
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
          const bool h1 = j + 512 < j_end, h2 = j + 1024 < j_end, h3 = j + 1536 < j_end;
          for (int p = 0; p < n_part; ++p) {
            const float* pp = part + static_cast<size_t>(p) * C + j;
            s0 += __ldcg(pp);
            if (h1) s1 += __ldcg(pp + 512);
            if (h2) s2 += __ldcg(pp + 1024);
            if (h3) s3 += __ldcg(pp + 1536);
          }
          scores[j] = s0;
          if (h1) scores[j + 512] = s1;
          if (h2) scores[j + 1024] = s2;
          if (h3) scores[j + 1536] = s3;
        }
        if (sm_tid == 0) counters[kc] = 0u;
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
    cudaError_t e = cudaFuncSetAttribute(profile_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PtCfg<false>::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(profile_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, PtCfg<true>::kSmem);
    return e;
  });
  if (attr != cudaSuccess) return cuda_error(attr, "profile_scores: smem attribute");
  const float scale_log2 = scale * 1.4426950408889634f;
  const dim3 grid(p.n_kc, Hkv, p.n_rg);
  unsigned int* status = device_status_ptr();
  {
    LaunchScope ls(KC_PROFILE, st);
    profile_tc_kernel<false><<<grid, kPtThreads, PtCfg<false>::kSmem, st>>>(
        tk, tq, q, nq, Hq, C, p.G, p.R, p.RT, p.n_rt, p.n_rg, p.tpc, p.n_kc, scale_log2, stats, part, cnt, scores, status);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "profile_scores: pass 1 launch");
  {
    LaunchScope ls(KC_PROFILE, st);
    e = launch_pdl(profile_tc_kernel<true>, grid, dim3(kPtThreads), PtCfg<true>::kSmem, st, tk, tq, q, nq, Hq, C, p.G, p.R,
                   p.RT, p.n_rt, p.n_rg, p.tpc, p.n_kc, scale_log2, stats, part, cnt, scores, status);
  }
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "profile_scores: pass 2 launch");
}

}  // namespace qcf
