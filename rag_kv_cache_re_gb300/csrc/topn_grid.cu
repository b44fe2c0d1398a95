// Exact top-N over many CTAs (one cooperative launch), for score vectors larger than one
// CTA's shared memory holds: the same selection as qcf_topn_select (the N largest,
// ties to the lower index, written ascending), with the scores read from global memory
// once, by all the CTAs at the same time.
//
// Each CTA keeps four scores per thread in registers (its slice of 4096) through every
// phase; the phases meet at grid barriers (bounded waits, so a CTA that never arrives
// turns into QCF_DEV_TIMEOUT instead of a hang; the cooperative launch guarantees every
// CTA is resident).  The scratch needs no clearing between calls: CTA 0 clears the
// counters and histograms and then publishes the call's 64-bit tag (a per-process
// sequence number), and every CTA waits for that tag before its first global update.
//   levels   histograms of 11, 11 and 10 key bits from the top, each restricted to the
//            bucket chosen so far, added into global bins; after each barrier every CTA
//            reads the bins and picks the bucket of the N-th largest key, until that
//            bucket holds at most kGridTarget keys
//   cands    each CTA appends its keys of that bucket, with their indices, to a global
//            candidate list
//   resolve  every CTA loads the candidates into shared memory and finishes the
//            selection there (the remaining key bits give K* and how many K*-valued keys
//            are taken; one warp ranks their indices when at most 32 keys equal K*, else
//            two 12-bit rounds over the indices give the last index taken)
//   output   each CTA publishes how many of its scores are taken; after the last barrier
//            it writes its taken indices, in order, at the sum of the counts before it
// When every key bit is fixed and still more than kGridCap keys equal K*, the CTAs
// publish their counts of greater and of equal keys instead and rank the equal ones
// by index across CTAs.
#include <atomic>
#include <chrono>

#include "qcf_internal.cuh"

namespace qcf {

constexpr int kGridThreads = 1024;
constexpr int kGridPer = 4;                               // scores per thread
constexpr int kGridSlice = kGridThreads * kGridPer;       // scores per CTA
constexpr int kGridCap = 16384;                           // candidates one CTA resolves in shared memory
constexpr int kGridTarget = 4096;                         // another global level while the bucket is larger
constexpr int kGridHistMax = 4096;                        // bins of the widest histogram (index rounds)
constexpr int kGridSmem = 2 * kGridCap * 4 + kGridHistMax * 4;   // candidate keys, indices, one histogram

// Workspace: [0] barrier arrivals, [1] candidate count, [2..3] the tag of the call that
// last cleared it, then the three levels' histograms (2048, 2048 and 1024 bins), the
// candidate list and per-CTA counts.
constexpr size_t kGridCtlWords = 64;
constexpr size_t kGridHistWords = 2048 + 2048 + 1024;
constexpr size_t kGridHeadBytes = (kGridCtlWords + kGridHistWords) * 4;   // control words and histograms

__device__ __forceinline__ unsigned int grid_order_key(float f) {
  unsigned int b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) == 0u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Barrier over the grid: the k-th barrier waits for k * gridDim.x arrivals.  The CTA's
// writes before it are ordered by the CTA barrier and released at GPU scope by thread 0's
// arrival; after it, the CTA reads other CTAs' data with L2 loads.  Returns false (every
// thread of the CTA) when the wait gave up.
__device__ bool grid_barrier(unsigned int* bar, unsigned int target, unsigned int* status, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
    const uint64_t t0 = globaltimer();
    bool ok = true;
    while (ld_acquire_u32(bar) < target) {
      if (globaltimer() - t0 > QCF_WAIT_NS) {
        ok = false;
        flag_status(status, QCF_DEV_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    *s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  return *s_ok != 0;
}

__device__ __forceinline__ unsigned int grid_scan_excl(unsigned int v, unsigned int* wsum, unsigned int* total) {
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

// out = {bin, still needed from it, the bin's count} for the need-th element from the top
// (desc) or bottom of h[nbins]; nbins a power of two from 512 to 8192.
__device__ void grid_pick_bin(const unsigned int* h, int nbins, bool desc, unsigned int need, unsigned int* wsum,
                              unsigned int* out) {
  const int k = nbins >= kGridThreads ? nbins / kGridThreads : 1;
  const int p0 = threadIdx.x * k;
  const int kk = p0 < nbins ? k : 0;   // threads past the last bin hold none
  unsigned int local = 0u;
  for (int i = 0; i < kk; ++i) local += h[desc ? nbins - 1 - (p0 + i) : p0 + i];
  unsigned int tot;
  unsigned int before = grid_scan_excl(local, wsum, &tot);
  if (before < need && need <= before + local) {
    for (int i = 0; i < kk; ++i) {
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

__device__ __forceinline__ int grid_level_shift(int lv) { return lv == 0 ? 21 : (lv == 1 ? 10 : 0); }
__device__ __forceinline__ int grid_level_bins(int lv) { return lv == 2 ? 1024 : 2048; }
__device__ __forceinline__ int grid_level_offset(int lv) { return lv * 2048; }

__global__ void __launch_bounds__(kGridThreads, 1)
    topn_grid_kernel(const float* __restrict__ scores, int C, int N, int32_t* __restrict__ sel,
                     unsigned int* __restrict__ ws, unsigned long long tag, unsigned int* status) {
  extern __shared__ __align__(16) unsigned int gsm[];
  unsigned int* ckey = gsm;                                  // [kGridCap]
  int* cidx = reinterpret_cast<int*>(gsm + kGridCap);        // [kGridCap]
  unsigned int* h = gsm + 2 * kGridCap;                      // [kGridHistMax]
  __shared__ unsigned int wsum[33];
  __shared__ unsigned int pick[3];
  __shared__ int s_ok;
  unsigned int* bar = ws;
  unsigned int* cand_n = ws + 1;
  unsigned long long* ready = reinterpret_cast<unsigned long long*>(ws + 2);
  unsigned int* ghist = ws + kGridCtlWords;                  // the levels' bins, back to back
  unsigned int* gkey = ws + kGridCtlWords + kGridHistWords;  // [kGridCap]
  int* gidx = reinterpret_cast<int*>(gkey + kGridCap);       // [kGridCap]
  unsigned int* counts = gkey + 2 * kGridCap;                // [gridDim.x][2]
  const int tid = threadIdx.x, lane = tid & 31;
  const unsigned int G = gridDim.x;
  unsigned int n_bar = 0;

  // this thread's four scores as keys, kept through every phase
  const int j0 = static_cast<int>(blockIdx.x) * kGridSlice + kGridPer * tid;
  unsigned int k[kGridPer];
  int n = 0;
  if (j0 + kGridPer <= C) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(scores + j0));
    k[0] = grid_order_key(f.x);
    k[1] = grid_order_key(f.y);
    k[2] = grid_order_key(f.z);
    k[3] = grid_order_key(f.w);
    n = kGridPer;
  } else {
    n = max(0, C - j0);
#pragma unroll
    for (int e = 0; e < kGridPer; ++e) k[e] = e < n ? grid_order_key(scores[j0 + e]) : 0u;
  }

  // ---- set-up: CTA 0 clears the counters and histograms, then publishes this call's tag
  if (blockIdx.x == 0) {
    for (size_t i = tid; i < kGridHistWords; i += kGridThreads) ghist[i] = 0u;
    if (tid == 0) {
      *bar = 0u;
      *cand_n = 0u;
    }
    __syncthreads();
    if (tid == 0) asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(ready), "l"(tag) : "memory");
  }

  // ---- levels
  unsigned int need = static_cast<unsigned int>(N), prefix = 0u, fmask = 0u, bucket = 0u;
  int lv = 0;
  while (true) {
    const int shift = grid_level_shift(lv), nb = grid_level_bins(lv);
    for (int i = tid; i < nb; i += kGridThreads) h[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kGridPer; ++e)
      if (e < n && (k[e] & fmask) == prefix) atomicAdd(&h[(k[e] >> shift) & (nb - 1)], 1u);
    if (lv == 0 && tid == 0) {   // the scratch is cleared for this call before the first global update
      const uint64_t t0 = globaltimer();
      bool ok = true;
      while (ld_acquire_u64(ready) != tag) {
        if (globaltimer() - t0 > QCF_WAIT_NS) {
          ok = false;
          flag_status(status, QCF_DEV_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
      s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    if (!s_ok) return;
    for (int i = tid; i < nb; i += kGridThreads)
      if (h[i]) atomicAdd(&ghist[grid_level_offset(lv) + i], h[i]);
    if (!grid_barrier(bar, (++n_bar) * G, status, &s_ok)) return;
    for (int i = tid; i < nb; i += kGridThreads) h[i] = __ldcg(&ghist[grid_level_offset(lv) + i]);
    __syncthreads();
    grid_pick_bin(h, nb, true, need, wsum, pick);
    prefix |= pick[0] << shift;
    fmask |= static_cast<unsigned int>(nb - 1) << shift;
    need = pick[1];
    bucket = pick[2];
    ++lv;
    if (bucket <= static_cast<unsigned int>(kGridTarget) || lv == 3) break;
  }

  const bool eq_mode = bucket > static_cast<unsigned int>(kGridCap);  // every bit fixed, too many equal keys
  unsigned int kstar = prefix, idx_star = 0u;
  if (!eq_mode) {
    // ---- candidates: this CTA's keys of the bucket, with their indices
#pragma unroll
    for (int e = 0; e < kGridPer; ++e) {
      const bool m = e < n && (k[e] & fmask) == prefix;
      const unsigned int bal = __ballot_sync(0xffffffffu, m);
      if (bal) {
        const int leader = __ffs(bal) - 1;
        unsigned int b0 = 0u;
        if (lane == leader) b0 = atomicAdd(cand_n, static_cast<unsigned int>(__popc(bal)));
        b0 = __shfl_sync(0xffffffffu, b0, leader);
        if (m) {
          const unsigned int pos = b0 + __popc(bal & ((1u << lane) - 1u));
          if (pos < static_cast<unsigned int>(kGridCap)) {
            gkey[pos] = k[e];
            gidx[pos] = j0 + e;
          }
        }
      }
    }
    if (!grid_barrier(bar, (++n_bar) * G, status, &s_ok)) return;
    // ---- resolve in shared memory (every CTA, the same result)
    const int n_c = min(static_cast<int>(ld_acquire_u32(cand_n)), kGridCap);
    for (int i = tid; i < n_c; i += kGridThreads) {
      ckey[i] = __ldcg(gkey + i);
      cidx[i] = __ldcg(gidx + i);
    }
    __syncthreads();
    unsigned int n_eq = bucket;   // keys in the current bucket; all equal K* once every bit is fixed
    for (; lv < 3; ++lv) {
      const int shift = grid_level_shift(lv), nb = grid_level_bins(lv);
      for (int i = tid; i < nb; i += kGridThreads) h[i] = 0u;
      __syncthreads();
      for (int i = tid; i < n_c; i += kGridThreads) {
        const unsigned int key = ckey[i];
        if ((key & fmask) == prefix) atomicAdd(&h[(key >> shift) & (nb - 1)], 1u);
      }
      __syncthreads();
      grid_pick_bin(h, nb, true, need, wsum, pick);
      prefix |= pick[0] << shift;
      fmask |= static_cast<unsigned int>(nb - 1) << shift;
      need = pick[1];
      n_eq = pick[2];
    }
    kstar = prefix;
    unsigned int ip = 0u, im = 0u;
    if (n_eq <= 32u) {
      // few keys equal K* (one, for most score vectors): one warp ranks their indices
      unsigned int* lst = h;        // [32] indices, then the count
      if (tid == 0) lst[32] = 0u;
      __syncthreads();
      for (int i = tid; i < n_c; i += kGridThreads)
        if (ckey[i] == kstar) {
          const unsigned int slot = atomicAdd(&lst[32], 1u);
          if (slot < 32u) lst[slot] = static_cast<unsigned int>(cidx[i]);
        }
      __syncthreads();
      if (tid < 32) {
        const unsigned int cnt = min(lst[32], 32u);
        const unsigned int mine_idx = static_cast<unsigned int>(tid) < cnt ? lst[tid] : 0xFFFFFFFFu;
        unsigned int rank = 0u;
        for (int j = 0; j < 32; ++j) rank += __shfl_sync(0xffffffffu, mine_idx, j) < mine_idx ? 1u : 0u;
        if (static_cast<unsigned int>(tid) < cnt && rank == need - 1u) pick[0] = mine_idx;
      }
      __syncthreads();
      ip = pick[0];
    }
    for (int il = 0; il < 2 && n_eq > 32u; ++il) {
      const int shift = il == 0 ? 12 : 0;
      for (int i = tid; i < 4096; i += kGridThreads) h[i] = 0u;
      __syncthreads();
      for (int i = tid; i < n_c; i += kGridThreads) {
        const unsigned int idx = static_cast<unsigned int>(cidx[i]);
        if (ckey[i] == kstar && (idx & im) == ip) atomicAdd(&h[(idx >> shift) & 4095u], 1u);
      }
      __syncthreads();
      grid_pick_bin(h, 4096, false, need, wsum, pick);
      ip |= pick[0] << shift;
      im |= 4095u << shift;
      need = pick[1];
    }
    idx_star = ip;
  }
  // ---- output: counts of taken (or of greater and equal) keys per CTA
  unsigned int f[kGridPer];
  unsigned int mine = 0u, mine_eq = 0u;
#pragma unroll
  for (int e = 0; e < kGridPer; ++e) {
    const bool gt = e < n && k[e] > kstar;
    const bool eq = e < n && k[e] == kstar;
    f[e] = eq_mode ? (gt ? 1u : (eq ? 2u : 0u))
                   : ((gt || (eq && static_cast<unsigned int>(j0 + e) <= idx_star)) ? 1u : 0u);
    mine += f[e] == 1u ? 1u : 0u;
    mine_eq += f[e] == 2u ? 1u : 0u;
  }
  unsigned int cta_taken, cta_eq;
  unsigned int r_taken = grid_scan_excl(mine, wsum, &cta_taken);
  unsigned int r_eq = grid_scan_excl(mine_eq, wsum, &cta_eq);
  if (tid == 0) {
    counts[2 * blockIdx.x] = cta_taken;
    counts[2 * blockIdx.x + 1] = cta_eq;
  }
  if (!grid_barrier(bar, (++n_bar) * G, status, &s_ok)) return;
  // offsets: taken keys (and, in eq mode, equal keys) of the CTAs before this one
  if (tid < 32) {
    unsigned int a = 0u, b = 0u;
    for (unsigned int c = lane; c < blockIdx.x; c += 32) {
      a += __ldcg(&counts[2 * c]);
      b += __ldcg(&counts[2 * c + 1]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if (lane == 0) {
      pick[0] = a;
      pick[1] = b;
    }
  }
  __syncthreads();
  const unsigned int before_taken = pick[0], before_eq = pick[1];
  unsigned int pos;
  if (!eq_mode) {
    pos = before_taken + r_taken;
  } else {
    // taken = every greater key and the first `need` keys equal to K* in index order; this
    // thread's first taken key follows the greater keys and the taken equal keys before it
    const unsigned int eq_before_me = before_eq + r_eq;
    pos = before_taken + r_taken + min(eq_before_me, need);
    unsigned int er = eq_before_me;
#pragma unroll
    for (int e = 0; e < kGridPer; ++e) {
      if (f[e] == 2u) {
        f[e] = er < need ? 1u : 0u;
        ++er;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < kGridPer; ++e)
    if (f[e] == 1u && pos < static_cast<unsigned int>(N)) sel[pos++] = j0 + e;
}

size_t topn_grid_workspace_size(int C) {
  const int G = (C + kGridSlice - 1) / kGridSlice;
  return kGridHeadBytes + static_cast<size_t>(2 * kGridCap) * 4 + static_cast<size_t>(2 * G) * 4 + 256;
}

static int topn_grid_capacity() {
  static PerDevice<int> max_grid;
  return max_grid.get(current_device(), [] {
    int per_sm = 0;
    if (cudaFuncSetAttribute(topn_grid_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGridSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topn_grid_kernel, kGridThreads, kGridSmem) != cudaSuccess)
      return 0;
    return per_sm * num_sms();
  });
}

int topn_grid_max_scores() {
  const long long n = static_cast<long long>(topn_grid_capacity()) * kGridSlice;
  return static_cast<int>(n < (1 << 24) ? n : (1 << 24));
}

// Call tags: a process-wide sequence under a high half drawn from the clock and an
// address, so a tag left in a workspace by an earlier call (or another process) never
// equals the current call's.
static unsigned long long next_call_tag() {
  static std::atomic<unsigned long long> seq{0};
  static const unsigned long long hi = [] {
    unsigned long long x = static_cast<unsigned long long>(
        std::chrono::steady_clock::now().time_since_epoch().count());
    x ^= reinterpret_cast<uintptr_t>(&seq) * 0x9E3779B97F4A7C15ull;
    x ^= x >> 29;
    return (x | 1ull) << 32;
  }();
  return hi ^ (seq.fetch_add(1) + 1);
}

qcf_status topn_grid_launch(const float* scores, int C, int N, int32_t* sel, void* ws, cudaStream_t st) {
  const int G = (C + kGridSlice - 1) / kGridSlice;
  const int cap = topn_grid_capacity();
  if (cap <= 0) return set_error(QCF_ERR_CUDA, "qcf_topn_select_ws: cooperative occupancy query failed");
  if (G > cap) return set_error(QCF_ERR_SHAPE, "qcf_topn_select_ws: %d scores need %d resident CTAs, at most %d", C, G, cap);
  unsigned int* w = static_cast<unsigned int*>(ws);
  unsigned long long tag = next_call_tag();
  unsigned int* status = device_status_ptr();
  void* args[] = {const_cast<float**>(&scores), &C, &N, &sel, &w, &tag, &status};
  LaunchScope ls(KC_TOPN, st);
  const cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<void*>(topn_grid_kernel), dim3(G),
                                                    dim3(kGridThreads), args, kGridSmem, st);
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_topn_select_ws: cooperative launch");
}

}  // namespace qcf
