// Dense GEMM on 5th-generation tensor cores: out = A * W^T with A [M][K] and
// W [N][K] bf16 (both K-major), fp32 accumulators in tensor memory (TMEM).
//
// Persistent, warp-specialised CTA of 6 warps, one CTA per SM:
//   warp 0   TMA producer: 128x64 A tile and BNx64 W tile per stage (128-byte swizzle)
//   warp 1   TMEM allocator and single-thread tcgen05.mma issuer (M=128, N=BN, K=16 steps)
//   warps 2-5 epilogue: tcgen05.ld of the accumulator (one row per thread), fused op, store
// The accumulator is double-buffered in TMEM so the epilogue of one tile overlaps
// the main loop of the next.  Work units are k ranges of (m tile, n tile); a CTA
// walks them on one of two schedules (UnitWalk): lockstep (units strided over the
// grid, m tile fastest, so concurrently running CTAs share each weight tile through
// L2; optionally k-split) or grouped stream-K (groups of tiles_m CTAs splitting the
// (n tile, k block) space evenly).  A tile shared by several units is finished by
// the last to arrive (counted with an atomic), which sums the fp32 partials in slot
// order -- deterministic -- and runs the epilogue; on the CTA's last unit it stages
// the partials (and, for the residual add, the x tile) in the idle pipeline stages.
//
// Fused epilogues:
//   STORE_BF16  out[m][n] = acc
//   ADD_F32     out[m][n] += acc                      (residual stream, fp32)
//   QKV_ROPE    columns are [q heads | k heads | v heads] of width D: q and k are
//               rotated by RoPE at rope_pos[m]; q goes to q_out[m], k/v are written
//               into the cache at row cache_row[m]
//   SWIGLU      W rows come in blocks of 64 gate rows then 64 up rows;
//               out[m][f] = silu(gate) * up
#include <algorithm>
#include <mutex>

#include "qcf_internal.cuh"

namespace qcf {

constexpr int kBM = 128, kBK = 64;
constexpr int kGemmThreads = 192;

template <int BN>
struct GemmCfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN >= 224 ? 4 : (BN == 128 ? 6 : 8);
  // two accumulator buffers; the allocation is a power of two (BN = 224 uses 448 of 512)
  static constexpr int TMEM_COLS = BN == 224 ? 512 : 2 * BN;
  static_assert(kBM * BN * 4 <= STAGES * STAGE_BYTES, "a residual tile must fit the stages");
  static constexpr int EPI_BYTES = 4 * 32 * 33 * 4;   // one 32x32 fp32 transpose tile per epilogue warp
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 /*barriers*/ + 1024 /*alignment slack*/;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Barrier over the 4 epilogue warps that also ORs a predicate across them.
__device__ __forceinline__ int epi_bar_or(int v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %1, 0;\n barrier.red.or.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"(v)
      : "memory");
  return static_cast<int>(out);
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    u.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    u.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    u.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    d[i] = u;
  }
}

// fp32 partial tiles in the workspace: each epilogue warp's 32 rows form one
// contiguous block of BN x 32 floats, column-quad-major inside it: element (row, col)
// of a 128 x BN slot sits at (((row / 32) * (BN / 4) + col / 4) * 32 + row % 32) * 4
// + col % 4.  A warp moving one float4 per lane touches 512 contiguous bytes, and a
// warp's whole partial is one bulk copy.
template <int BN>
__device__ __forceinline__ size_t part_idx(int row, int quad) {
  return ((static_cast<size_t>(row >> 5) * (BN / 4) + quad) * 32 + (row & 31)) * 4;
}

// Loads 32 accumulator columns [32c, 32c+32) of this thread's row, either from
// TMEM (direct) or as the in-order sum of the split-K partials in the workspace.
template <int BN>
struct ChunkLoader {
  uint32_t taddr;       // TMEM address of (row quarter, column 0) of the accumulator
  const float* part;    // the tile's first partial slot, or nullptr for TMEM
  const float* rest;    // its second partial slot; the later ones follow at part_stride
  int splits;           // partial slots to sum
  size_t part_stride;   // floats between consecutive slots after the first
  int row;              // row within the tile
  __device__ __forceinline__ void operator()(int c, float* v) const {
    if (part == nullptr) {
      tmem_ld32(taddr + static_cast<uint32_t>(c * 32), v);
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 t = __ldcg(reinterpret_cast<const float4*>(part + part_idx<BN>(row, c * 8 + q)));
        v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
      }
      // two slots per round trip (the sum stays in slot order)
      int s = 1;
#pragma unroll 1
      for (; s + 1 < splits; s += 2) {
        const float* p = rest + static_cast<size_t>(s - 1) * part_stride;
        float4 t0[8], t1[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          t0[q] = __ldcg(reinterpret_cast<const float4*>(p + part_idx<BN>(row, c * 8 + q)));
          t1[q] = __ldcg(reinterpret_cast<const float4*>(p + part_stride + part_idx<BN>(row, c * 8 + q)));
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          v[4 * q] += t0[q].x; v[4 * q + 1] += t0[q].y; v[4 * q + 2] += t0[q].z; v[4 * q + 3] += t0[q].w;
          v[4 * q] += t1[q].x; v[4 * q + 1] += t1[q].y; v[4 * q + 2] += t1[q].z; v[4 * q + 3] += t1[q].w;
        }
      }
      if (s < splits) {
        const float* p = rest + static_cast<size_t>(s - 1) * part_stride;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(p + part_idx<BN>(row, c * 8 + q)));
          v[4 * q] += t.x; v[4 * q + 1] += t.y; v[4 * q + 2] += t.z; v[4 * q + 3] += t.w;
        }
      }
    }
  }
};

// The last arriver's partial sums with the other units' partials staged in shared
// memory: slot j of the tile (in slot order) is this unit's own accumulator in TMEM
// when j == own, else staged part jj = j - (j > own) at smem[((jj * BN/4 + quad) * 32
// + lane) * 4] (a warp's 32 rows of one column quad, as stored in the workspace).
// Summing in slot order keeps the result independent of which unit arrives last.
template <int BN>
struct StagedPartLoader {
  uint32_t taddr;
  const float* smem;  // this warp's staged parts
  int parts, own;
  __device__ __forceinline__ void operator()(int c, float* v) const {
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int j = 0; j < parts; ++j) {
      if (j == own) {
        if (j == 0) {
          tmem_ld32(taddr + static_cast<uint32_t>(c * 32), v);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float t[16];
            tmem_ld16(taddr + static_cast<uint32_t>(c * 32 + h * 16), t);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[h * 16 + i] += t[i];
          }
        }
      } else {
        const float4* src = reinterpret_cast<const float4*>(smem) + (j - (j > own)) * (BN / 4) * 32 + c * 8 * 32 + lane;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 x = src[q * 32];
          if (j == 0) {
            v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
          } else {
            v[4 * q] += x.x; v[4 * q + 1] += x.y; v[4 * q + 2] += x.z; v[4 * q + 3] += x.w;
          }
        }
      }
    }
  }
};

__device__ __forceinline__ void rope_pair32(float* lo, float* hi, const float* cs, const float* sn) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float a = lo[i], b = hi[i];
    lo[i] = a * cs[i] - b * sn[i];
    hi[i] = b * cs[i] + a * sn[i];
  }
}

__device__ __forceinline__ void load_f32x(const float* src, float* v, int n) {
  for (int i = 0; i < n; i += 4) {
    const float4 t = *reinterpret_cast<const float4*>(src + i);
    v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
  }
}

// Epilogue of one tile for the calling thread's row.  `row` < M is checked here.
// `tile` is this warp's 32x33 fp32 staging area in shared memory.
template <int BN, int EPI, int HD, class Loader>
__device__ __forceinline__ void tile_epilogue(const Loader& ld, const EpiParams& ep, int row, int M, int n0,
                                              float* tile) {
  const bool live = row < M;
  if constexpr (EPI == EPI_STORE_BF16) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(ep.out);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float v[32];
      ld(c, v);
      if (live) store_bf16x32(out + static_cast<size_t>(row) * ep.ldo + n0 + c * 32, v);
    }
  } else if constexpr (EPI == EPI_ADD_F32) {
    // The accumulator arrives one row per thread; the residual x is read and
    // written with 4 full 128-byte row segments per warp instruction by passing
    // each 32x32 chunk through shared memory.  x of the next chunk is loaded
    // ahead while the current one is transposed and added.
    const int lane = threadIdx.x & 31;
    const int row0 = row - lane;                 // first row of this warp's 32
    const int rr = lane >> 3, cq = (lane & 7) * 4;
    float* out = static_cast<float*>(ep.out);
    auto xptr = [&](int c, int i) {
      return reinterpret_cast<float4*>(out + static_cast<size_t>(row0 + i * 4 + rr) * ep.ldo + n0 + c * 32 + cq);
    };
    auto row_ok = [&](int i) { return row0 + i * 4 + rr < M; };
    // chunks of this tile inside the row (all of them but in a ragged last column tile)
    const int nch = min(BN / 32, (ep.ldo - n0) / 32);
    float4 xa[8], xb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (row_ok(i)) xa[i] = *xptr(0, i);
    auto add_store = [&](int c, const float4* xr) {
      float v[32];
      ld(c, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) tile[lane * 33 + j] = v[j];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float* tr = tile + (i * 4 + rr) * 33 + cq;
        if (row_ok(i)) {
          float4 t = xr[i];
          t.x += tr[0]; t.y += tr[1]; t.z += tr[2]; t.w += tr[3];
          *xptr(c, i) = t;
        }
      }
      __syncwarp();
    };
#pragma unroll 1
    for (int c = 0; c < nch; c += 2) {
      if (c + 1 < nch) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (row_ok(i)) xb[i] = *xptr(c + 1, i);
      }
      add_store(c, xa);
      if (c + 2 < nch) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (row_ok(i)) xa[i] = *xptr(c + 2, i);
      }
      if (c + 1 < nch) add_store(c + 1, xb);
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(ep.out);
    const int f0 = n0 / 2;
#pragma unroll 1
    for (int blk = 0; blk < BN / 128; ++blk) {
#pragma unroll 1
      for (int j = 0; j < 2; ++j) {
        float g[32], u[32];
        ld(blk * 4 + j, g);
        ld(blk * 4 + 2 + j, u);
        if (live) {
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] = g[i] / (1.0f + __expf(-g[i])) * u[i];
          store_bf16x32(out + static_cast<size_t>(row) * ep.ldo + f0 + blk * 64 + j * 32, g);
        }
      }
    }
  } else {  // EPI_QKV_ROPE
    static_assert(HD == 16 || HD == 64 || HD == 128, "head dim");
    static_assert(BN % HD == 0, "tile must hold whole heads");
    const int qw = ep.Hq * HD, kw = ep.Hkv * HD;
    int p = 0, crow = 0;
    bool kv_ok = true;
    if (live) {
      p = ep.rope_pos[row];
      crow = ep.cache_row ? ep.cache_row[row] : 0;
      if (static_cast<unsigned>(p) >= static_cast<unsigned>(ep.max_pos)) {
        flag_status(ep.status, QCF_DEV_BAD_INDEX);
        p = 0;
      }
      if (static_cast<unsigned>(crow) >= static_cast<unsigned>(ep.T)) {
        flag_status(ep.status, QCF_DEV_BAD_INDEX);
        kv_ok = false;
      }
    }
    const float* cs_row = ep.cos_t + static_cast<size_t>(p) * (HD / 2);
    const float* sn_row = ep.sin_t + static_cast<size_t>(p) * (HD / 2);
#pragma unroll 1
    for (int h = 0; h < BN / HD; ++h) {
      const int col = n0 + h * HD;  // first global column of this head
      __nv_bfloat16* dst = nullptr;
      bool rotate = true;
      const bool dst_is_q = col < qw;
      if (col < qw) {
        dst = ep.q_out + static_cast<size_t>(row) * qw + col;
      } else if (col < qw + kw) {
        dst = ep.k_cache + static_cast<size_t>(crow) * kw + (col - qw);
      } else {
        dst = ep.v_cache + static_cast<size_t>(crow) * kw + (col - qw - kw);
        rotate = false;
      }
      if constexpr (HD >= 64) {
        constexpr int dist = HD / 64;  // chunks between element k and k + D/2
#pragma unroll 1
        for (int j = 0; j < dist; ++j) {
          float lo[32], hi[32];
          const int c_lo = h * (HD / 32) + j;
          ld(c_lo, lo);
          ld(c_lo + dist, hi);
          if (live && (dst_is_q || kv_ok)) {
            if (rotate) {
              float cs[32], sn[32];
              load_f32x(cs_row + j * 32, cs, 32);
              load_f32x(sn_row + j * 32, sn, 32);
              rope_pair32(lo, hi, cs, sn);
            }
            store_bf16x32(dst + j * 32, lo);
            store_bf16x32(dst + HD / 2 + j * 32, hi);
          }
        }
      } else {  // HD == 16: one chunk holds two heads; handle them when h is even
        if (h & 1) continue;
        float v[32];
        ld(h / 2, v);
        if (live) {
          float cs[8], sn[8];
          load_f32x(cs_row, cs, 8);
          load_f32x(sn_row, sn, 8);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int colh = col + hh * 16;
            if (colh >= qw && !kv_ok) continue;
            bool rot = true;
            __nv_bfloat16* d2;
            if (colh < qw) {
              d2 = ep.q_out + static_cast<size_t>(row) * qw + colh;
            } else if (colh < qw + kw) {
              d2 = ep.k_cache + static_cast<size_t>(crow) * kw + (colh - qw);
            } else {
              d2 = ep.v_cache + static_cast<size_t>(crow) * kw + (colh - qw - kw);
              rot = false;
            }
            float o[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float a = v[hh * 16 + i], b = v[hh * 16 + 8 + i];
              o[i] = rot ? a * cs[i] - b * sn[i] : a;
              o[8 + i] = rot ? b * cs[i] + a * sn[i] : b;
            }
            uint4* dd = reinterpret_cast<uint4*>(d2);
            uint4 u0, u1;
            u0.x = pack_bf16x2(o[0], o[1]); u0.y = pack_bf16x2(o[2], o[3]);
            u0.z = pack_bf16x2(o[4], o[5]); u0.w = pack_bf16x2(o[6], o[7]);
            u1.x = pack_bf16x2(o[8], o[9]); u1.y = pack_bf16x2(o[10], o[11]);
            u1.z = pack_bf16x2(o[12], o[13]); u1.w = pack_bf16x2(o[14], o[15]);
            dd[0] = u0;
            dd[1] = u1;
          }
        }
      }
    }
  }
}

// Residual add of one warp's 32 rows with everything staged in shared memory (the
// pipeline stages, idle on the CTA's last unit).  Lane 0 loads the warp's x rows as
// BN/32 TMA boxes of 32 rows x 32 fp32 (128-byte swizzle: row r keeps 16-byte
// chunk j at j ^ (r % 8), so row-per-lane float4 accesses hit every bank once), and
// lanes 1.. bulk-copy the other units' partials of a shared tile.  The accumulator
// sum (slot order, this unit's own part from TMEM) is added into x in place and the
// boxes are stored back by TMA, which leaves rows past M untouched.  All copies
// complete on bar (one use per launch).
template <int BN>
__device__ __forceinline__ void add_tile_staged(uint32_t taddr, const CUtensorMap* tmX, uint8_t* region,
                                                const float* first, const float* rest, size_t step, int parts,
                                                int own, uint64_t* bar, uint32_t phase, int row0, int n0,
                                                unsigned int* status, int nbox) {
  constexpr int kBox = 32 * 32 * 4;            // one x box
  constexpr int kPart = BN * 32 * 4;           // a warp's rows of one partial
  const int lane = threadIdx.x & 31;
  float* xs = reinterpret_cast<float*>(region);
  const float* ps = reinterpret_cast<const float*>(region + (BN / 32) * kBox);
  // nbox: the x boxes inside the row (fewer than BN / 32 only in a ragged last column tile)
  if (lane == 0) {
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbox * kBox + (parts - 1) * kPart));
#pragma unroll 1
    for (int c = 0; c < nbox; ++c) tma_load_2d(xs + c * 1024, tmX, bar, n0 + c * 32, row0);
  }
  __syncwarp();
  if (parts > 1 && lane < parts && lane != own) {
    const float* src = lane == 0 ? first : rest + (lane - 1) * step;
    bulk_load_g2s(region + (BN / 32) * kBox + (lane - (lane > own)) * kPart, src, kPart, bar);
  }
  if (!mbar_wait(bar, phase)) {
    flag_status(status, QCF_DEV_TIMEOUT);
    mbar_wait(bar, phase);  // once more, bounded, so no copy is left landing in smem
    return;
  }
#pragma unroll 1
  for (int c = 0; c < nbox; ++c) {
    float v[32];
    if (parts == 1) {
      tmem_ld32(taddr + static_cast<uint32_t>(c * 32), v);
    } else {
#pragma unroll 1
      for (int j = 0; j < parts; ++j) {
        if (j == own) {
          if (j == 0) {
            tmem_ld32(taddr + static_cast<uint32_t>(c * 32), v);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float t[16];
              tmem_ld16(taddr + static_cast<uint32_t>(c * 32 + h * 16), t);
#pragma unroll
              for (int i = 0; i < 16; ++i) v[h * 16 + i] += t[i];
            }
          }
        } else {
          const float4* src = reinterpret_cast<const float4*>(ps) + (j - (j > own)) * (BN / 4) * 32 + c * 8 * 32 + lane;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 x = src[q * 32];
            if (j == 0) {
              v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
            } else {
              v[4 * q] += x.x; v[4 * q + 1] += x.y; v[4 * q + 2] += x.z; v[4 * q + 3] += x.w;
            }
          }
        }
      }
    }
    float4* row = reinterpret_cast<float4*>(xs + c * 1024 + lane * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4 t = row[q ^ (lane & 7)];
      t.x += v[4 * q]; t.y += v[4 * q + 1]; t.z += v[4 * q + 2]; t.w += v[4 * q + 3];
      row[q ^ (lane & 7)] = t;
    }
  }
  fence_proxy_async_smem();  // the generic-proxy writes above, before TMA reads them
  __syncwarp();
  if (lane == 0) {
#pragma unroll 1
    for (int c = 0; c < nbox; ++c) tma_store_2d(tmX, xs + c * 1024, n0 + c * 32, row0);
    bulk_commit_group();
    bulk_wait_group0();
  }
  __syncwarp();
}

// One pass of a shared tile's staged fixup for the store / SwiGLU / QKV epilogues:
// columns [h BNP, (h + 1) BNP) of the tile.  The other units' partials of those columns
// (a contiguous BNP x 32-float block of each warp's slab) are bulk-copied to smem, then
// the epilogue runs on their slot-ordered sum with this unit's own TMEM part.
template <int BNP, int EPI, int HD>
__device__ __forceinline__ bool staged_fixup_pass(int h, uint32_t taddr, float* sp, const float* first,
                                                  const float* rest, size_t step, int parts, int own, uint64_t* bar,
                                                  const EpiParams& ep, int row, int M, int n0, float* tile,
                                                  unsigned int* status) {
  constexpr int kPassPart = BNP * 32 * 4;  // a warp's rows of one partial, these columns
  const int lane = threadIdx.x & 31;
  if (h > 0) {
    fence_proxy_async_smem();  // the previous pass's generic reads, before these copies overwrite them
    __syncwarp();
  }
  if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>((parts - 1) * kPassPart));
  __syncwarp();
  if (lane < parts && lane != own) {
    const float* src = (lane == 0 ? first : rest + (lane - 1) * step) + static_cast<size_t>(h) * BNP * 32;
    bulk_load_g2s(sp + static_cast<size_t>(lane - (lane > own)) * (kPassPart / 4), src, kPassPart, bar);
  }
  if (!mbar_wait(bar, static_cast<uint32_t>(h & 1))) {
    flag_status(status, QCF_DEV_TIMEOUT);
    mbar_wait(bar, static_cast<uint32_t>(h & 1));  // once more, bounded, so no copy is left landing in smem
    return false;
  }
  tc_fence_after();
  StagedPartLoader<BNP> ld{taddr + static_cast<uint32_t>(h * BNP), sp, parts, own};
  tile_epilogue<BNP, EPI, HD>(ld, ep, row, M, n0 + h * BNP, tile);
  return true;
}

// One work unit: k blocks [kb0, kb1) of output tile (mt, nt).  A tile whose k range
// is shared by several units (parts > 1) is finished by whichever arrives last: each
// writes its fp32 partial and bumps the tile's counter, and the last one sums the
// partials in order and runs the epilogue (no unit ever waits for another).  Partial
// slots are numbered in units of one slot (128 or 256 rows x BN floats).
struct Unit {
  int mt, nt, kb0, kb1;
  int parts;   // units sharing the tile (1: this unit has the whole k range)
  int cnt;     // arrival counter of the tile
  int mine;    // this unit's partial slot
  int first;   // the tile's first partial slot ...
  int rest;    // ... its second; later ones follow every `step` slots
  int step;
};

// The units one CTA works through, in order.  Two schedules:
//  * lockstep (groups == 0): unit u = blockIdx.x + i * gridDim.x over tiles x splits,
//    m tile fastest, so the CTAs running together share each weight tile's k walk;
//  * grouped stream-K (groups > 0): CTA b computes m tile b % tiles_m for group
//    b / tiles_m, and group g owns iterations [g I / G, (g + 1) I / G) of the
//    (n tile, k block) space (I = tiles_n x kb_total, G groups).  The tiles_m CTAs of
//    a group walk the same weight blocks side by side (one HBM read of each serves
//    all m tiles), and every CTA gets the same number of k blocks whatever the tile
//    count, so no last round runs part-empty.  A column cut by a group boundary is
//    shared: a group's piece of it is its first (slot 0) or last (slot 1) piece.
// The host keeps I x G below 2^31.
struct UnitWalk {
  int tiles_m, kb_total, splits, units, groups;
  int u, mt, g, total, x, xend;

  __device__ void init(int tm, int tn, int kbt, int sp, int gr) {
    tiles_m = tm; kb_total = kbt; splits = sp; groups = gr;
    units = tm * tn * sp;
    u = blockIdx.x;
    mt = static_cast<int>(blockIdx.x) % tm;
    g = static_cast<int>(blockIdx.x) / tm;
    total = tn * kbt;
    x = gr > 0 ? start_of(g) : 0;
    xend = gr > 0 ? start_of(g + 1) : 0;
  }
  __device__ int start_of(int grp) const { return grp * total / groups; }
  // the group whose range holds iteration it: the largest grp with start_of(grp) <= it
  __device__ int owner(int it) const { return ((it + 1) * groups + total - 1) / total - 1; }
  __device__ int slot(int grp, int which) const { return (grp * tiles_m + mt) * 2 + which; }

  __device__ bool next(Unit& w) {
    if (groups == 0) {
      if (u >= units) return false;
      w.mt = u % tiles_m;
      const int r = u / tiles_m;
      const int sp = r % splits;
      w.nt = r / splits;
      w.kb0 = static_cast<int>(static_cast<long long>(kb_total) * sp / splits);
      w.kb1 = static_cast<int>(static_cast<long long>(kb_total) * (sp + 1) / splits);
      w.parts = splits;
      w.cnt = w.nt * tiles_m + w.mt;
      w.first = w.cnt * splits;
      w.mine = w.first + sp;
      w.rest = w.first + 1;
      w.step = 1;
      u += gridDim.x;
      return true;
    }
    if (x >= xend) return false;
    const int nt = x / kb_total;
    const int c0 = nt * kb_total;
    const int lim = xend < c0 + kb_total ? xend : c0 + kb_total;
    w.mt = mt;
    w.nt = nt;
    w.kb0 = x - c0;
    w.kb1 = lim - c0;
    const int fg = owner(c0), lg = owner(c0 + kb_total - 1);
    w.parts = lg - fg + 1;
    w.cnt = nt * tiles_m + mt;
    w.mine = slot(g, start_of(g) >= c0 ? 0 : 1);
    w.first = slot(fg, start_of(fg) >= c0 ? 0 : 1);
    w.rest = slot(fg + 1, 0);  // later contributors start inside the column: their slot 0
    w.step = 2 * tiles_m;
    x = lim;
    return true;
  }
};

template <int BN, int EPI, int HD, bool BMN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmX, int M, int N, int K, int splits, int groups,
                        const EpiParams ep, float* __restrict__ ws_part,
                        unsigned int* __restrict__ ws_cnt, unsigned int* status) {
  using Cfg = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::STAGES * Cfg::STAGE_BYTES);
  uint64_t* empty = full + Cfg::STAGES;
  uint64_t* tfull = empty + Cfg::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* xbar = tempty + 2;  // one per epilogue warp: its staged residual rows landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 4);
  volatile int* s_last = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* epi_tiles = reinterpret_cast<float*>(smem + Cfg::STAGES * Cfg::STAGE_BYTES + 1024);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_m = (M + kBM - 1) / kBM;
  const int tiles_n = (N + BN - 1) / BN;  // BN = 224: the last column tile is ragged
  const int kb_total = K / kBK;
  UnitWalk walk;
  walk.init(tiles_m, tiles_n, kb_total, splits, groups);
  constexpr size_t kSlot = static_cast<size_t>(kBM) * BN;  // floats of one partial slot

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    for (int q = 0; q < 4; ++q) mbar_init(&xbar[q], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      auto load_w = [&](uint8_t* a_s, int kb, int nt, uint64_t* bar) {
        if constexpr (BMN) {   // W stored [K][N]: BN/64 boxes of 64 K rows x 64 N columns
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(a_s + Cfg::A_BYTES + j * (kBK * 128), &tmB, bar, nt * BN + j * 64, kb * kBK);
        } else {
          tma_load_2d(a_s + Cfg::A_BYTES, &tmB, bar, kb * kBK, nt * BN);
        }
      };
      // The weights are never written by the kernels a programmatic launch overlaps,
      // so the first unit's weight stages are requested before waiting for them;
      // the activation half of each of those stages follows the wait.
      int npre = 0;
      {
        UnitWalk peek = walk;
        Unit w0;
        if (peek.next(w0)) {
          npre = min(Cfg::STAGES, w0.kb1 - w0.kb0);
          for (int j = 0; j < npre; ++j) {
            mbar_arrive_expect_tx(&full[j], Cfg::STAGE_BYTES);
            load_w(smem + j * Cfg::STAGE_BYTES, w0.kb0 + j, w0.nt, &full[j]);
          }
        }
      }
      pdl_wait();
      pdl_launch_dependents();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int issued = 0;  // k blocks loaded so far; the first npre had their weights requested above
      Unit w;
      while (ok && walk.next(w)) {
        const int mt = w.mt, nt = w.nt;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++issued) {
          uint8_t* a_s = smem + stage * Cfg::STAGE_BYTES;
          if (issued >= npre) {
            if (!mbar_wait(&empty[stage], phase ^ 1u)) {
              flag_status(status, QCF_DEV_TIMEOUT);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
            load_w(a_s, kb, nt, &full[stage]);
          }
          tma_load_2d(a_s, &tmA, &full[stage], kb * kBK, mt * kBM);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, BMN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Unit w;
      for (int local = 0; ok && walk.next(w); ++local) {
        const int kb0 = w.kb0, kb1 = w.kb1;
        const int acc = local & 1;
        if (!mbar_wait(&tempty[acc], ((local >> 1) & 1) ^ 1u)) {
          flag_status(status, QCF_DEV_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase)) {
            flag_status(status, QCF_DEV_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * Cfg::STAGE_BYTES);
          const uint32_t b_addr = a_addr + Cfg::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // K-major: 16 K elements are 32 bytes along the swizzled row; MN-major:
            // 16 K indices are two 1024-byte atoms
            const uint64_t bdesc = BMN ? sdesc_mnmajor_sw128(b_addr + kk * 2048, kBK * 128)
                                       : sdesc_kmajor_sw128(b_addr + kk * 32);
            umma_f16(d_tmem, sdesc_kmajor_sw128(a_addr + kk * 32), bdesc, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == Cfg::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
      }
    }
  } else {
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    float* my_tile = epi_tiles + (warp - 2) * (32 * 33);
    pdl_wait();  // the residual, position tables and output buffers come from earlier kernels
    pdl_launch_dependents();
    // shared tiles go through epilogue-wide barriers: with any, abort only together
    const bool shared_tiles = splits > 1 || groups > 0;
    Unit w;
    for (int local = 0; walk.next(w); ++local) {
      const int mt = w.mt, nt = w.nt;
      const int acc = local & 1;
      if constexpr (EPI == EPI_ADD_F32) {
        // the residual rows of the CTA's last unit: pull them into L2 (kept there
        // ahead of the weight stream) while the main loop runs.  Only for GEMMs of up to
        // 2048 rows: with many m tiles the kept lines cost the weight reuse more than
        // they save (measured on the 5184-row full prefill).
        UnitWalk peek = walk;
        Unit nx;
        const int r = mt * kBM + row_in_tile;
        if (M <= 2048 && !peek.next(nx) && r < M) {
          const char* xr = reinterpret_cast<const char*>(static_cast<const float*>(ep.out) + static_cast<size_t>(r) * ep.ldo +
                                                         static_cast<size_t>(nt) * BN);
          const int row_bytes = min(BN, N - nt * BN) * 4;
#pragma unroll 1
          for (int b = 0; b < row_bytes; b += 128) asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(xr + b));
        }
      }
      const bool got = mbar_wait(&tfull[acc], (local >> 1) & 1);
      if (!got) flag_status(status, QCF_DEV_TIMEOUT);
      if (shared_tiles) {
        if (epi_bar_or(!got)) break;
      } else if (!got) {
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quarter * 32) << 16);
      const int row = mt * kBM + row_in_tile;
      const int n0 = nt * BN;
      // On the CTA's last unit no stage will be loaded again and the MMAs that read
      // them have completed (tfull): the residual-add epilogue stages there.
      bool last_unit = false;
      {
        UnitWalk peek = walk;
        Unit nx;
        last_unit = !peek.next(nx);
      }
      const bool warp_live = row - lane < M;  // rows past M are neither written nor summed
      bool staged = false;
      if constexpr (EPI == EPI_ADD_F32) staged = w.parts == 1 && last_unit;
      if (staged) {
        if (warp_live)
          add_tile_staged<BN>(taddr, &tmX, smem + static_cast<size_t>(quarter) * BN * 32 * 4, nullptr, nullptr, 0, 1, 0,
                              &xbar[quarter], 0, row - lane, n0, status, min(BN, N - n0) / 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      } else if (w.parts == 1) {
        ChunkLoader<BN> ld{taddr, nullptr, nullptr, 1, 0, row_in_tile};
        tile_epilogue<BN, EPI, HD>(ld, ep, row, M, n0, my_tile);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      } else {
        // On the CTA's last unit the pipeline stages are idle and this unit's own
        // accumulator stays in TMEM: the last arriver stages the other partials there
        // (one bulk copy per partial and warp; the residual add stages x beside them)
        // and sums from shared memory.  Warp regions are laid out for the live warps
        // only; a tile whose staging does not fit goes in two passes of BN / 2 columns.
        constexpr int kWarpPartBytes = BN * 32 * 4;  // a warp's rows of one partial (or its x rows)
        const int per_warp = (EPI == EPI_ADD_F32 ? w.parts : w.parts - 1) * kWarpPartBytes;
        const int live_warps = min(4, (M - mt * kBM + 31) / 32);
        constexpr int kStageBytes = Cfg::STAGES * Cfg::STAGE_BYTES;
        int passes = 0;
        if (last_unit && w.parts <= 32) {
          if (live_warps * per_warp <= kStageBytes) passes = 1;
          else if (BN == 256 && live_warps * (per_warp / 2) <= kStageBytes) passes = 2;
        }
        const bool stage = passes > 0;
        // When staging is possible and every other unit of the tile has already arrived
        // (the usual case under stream-K: the other pieces of a cut column come first
        // in their groups' ranges), this unit is the last: it writes no partial.
        // the accumulator goes back to the MMA warp as soon as nothing reads it any more:
        // after the partial is written, or after a staged fixup that reads it in TMEM
        bool released = false;
        auto release_acc = [&] {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
          released = true;
        };
        int last = 0;
        if (stage) {
          if (threadIdx.x == 64) {
            unsigned int c;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(&ws_cnt[w.cnt]) : "memory");
            const int all_in = c == static_cast<unsigned int>(w.parts - 1);
            if (all_in) ws_cnt[w.cnt] = 0u;  // no other unit of the tile remains: back to zero
            *s_last = all_in;
          }
          epi_bar();
          last = *s_last;
          epi_bar();
        }
        if (!last) {
          float* mine = ws_part + static_cast<size_t>(w.mine) * kSlot;
#pragma unroll 1
          for (int c = 0; c < (warp_live ? BN / 32 : 0); ++c) {
            float v[32];
            tmem_ld32(taddr + static_cast<uint32_t>(c * 32), v);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<float4*>(mine + part_idx<BN>(row_in_tile, c * 8 + q)) =
                  make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
          if (!stage) release_acc();
          __threadfence();
          epi_bar();
          if (threadIdx.x == 64) {
            const unsigned int prev = atomicAdd(&ws_cnt[w.cnt], 1u);
            const int is_last = prev == static_cast<unsigned int>(w.parts - 1);
            if (is_last) ws_cnt[w.cnt] = 0u;  // back to zero for the next launch on this workspace
            *s_last = is_last;
          }
          epi_bar();
          last = *s_last;
          epi_bar();
        }
        if (!(last && warp_live) && !released) release_acc();
        if (last && warp_live) {
          __threadfence();
          const int own = w.mine == w.first ? 0 : (w.mine - w.rest) / w.step + 1;
          float* sp = reinterpret_cast<float*>(smem + static_cast<size_t>(quarter) * (per_warp / max(passes, 1)));
          const float* pfirst = ws_part + static_cast<size_t>(w.first) * kSlot + part_idx<BN>(quarter * 32, 0);
          const float* prest = ws_part + static_cast<size_t>(w.rest) * kSlot + part_idx<BN>(quarter * 32, 0);
          if (stage) {
            // the other units' partials were written with generic stores: order the
            // async-proxy (bulk copy) reads below after them
            asm volatile("fence.proxy.async;" ::: "memory");
            tc_fence_after();
            if constexpr (EPI == EPI_ADD_F32) {
              if (passes == 1) {
                add_tile_staged<BN>(taddr, &tmX, reinterpret_cast<uint8_t*>(sp), pfirst, prest, w.step * kSlot, w.parts,
                                    own, &xbar[quarter], 0, row - lane, n0, status, min(BN, N - n0) / 32);
              } else if constexpr (BN == 256) {
#pragma unroll 1
                for (int h = 0; h < 2; ++h)
                  add_tile_staged<BN / 2>(taddr + static_cast<uint32_t>(h * BN / 2), &tmX, reinterpret_cast<uint8_t*>(sp),
                                          pfirst + h * (BN / 2) * 32, prest + h * (BN / 2) * 32, w.step * kSlot,
                                          w.parts, own, &xbar[quarter], static_cast<uint32_t>(h), row - lane,
                                          n0 + h * (BN / 2), status, min(BN / 2, N - n0 - h * (BN / 2)) / 32);
              }
            } else {
              if (passes == 1) {
                staged_fixup_pass<BN, EPI, HD>(0, taddr, sp, pfirst, prest, w.step * kSlot, w.parts, own,
                                               &xbar[quarter], ep, row, M, n0, my_tile, status);
              } else if constexpr (BN == 256) {
#pragma unroll 1
                for (int h = 0; h < 2; ++h)
                  if (!staged_fixup_pass<BN / 2, EPI, HD>(h, taddr, sp, pfirst, prest, w.step * kSlot, w.parts, own,
                                                          &xbar[quarter], ep, row, M, n0, my_tile, status))
                    break;
              }
            }
          }
          if (!stage) {
            ChunkLoader<BN> ld{0u, ws_part + static_cast<size_t>(w.first) * kSlot,
                           ws_part + static_cast<size_t>(w.rest) * kSlot, w.parts, w.step * kSlot, row_in_tile};
            tile_epilogue<BN, EPI, HD>(ld, ep, row, M, n0, my_tile);
          }
          if (!released) release_acc();
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

struct GemmPlan {
  int BN;
  int splits;
  int tiles;
  int groups;  // > 0: grouped stream-K with this many groups of tiles_m CTAs
};

// Arrival counters sit at the front of the workspace, one per output tile, and every
// launch leaves them zero; a plan that shares tiles needs tiles <= kCntCells.
constexpr int kCntCells = 4096;
constexpr size_t kCntBytes = kCntCells * sizeof(unsigned int);

// Main-loop k blocks a grouped stream-K plan must save over the lockstep grid before
// its shared-tile fixups pay off, fitted to 16 layer-shape x M measurements on GB300
// (M = 256 ... 1664): 40, plus 13 per partial beyond two.
constexpr int kSkMinGain = 40;
constexpr int kSkGainPerPart = 13;

// Chooses the tile width BN, the k split and the schedule from measurements on GB300:
//  * M > 128 (the recompute GEMMs): the widest tile (BN = 256).  The lockstep grid
//    runs ceil(tiles / SMs) rounds of a whole k range each; grouped stream-K gives
//    every CTA (SMs / tiles_m groups of tiles_m CTAs) an equal share of the
//    (n tile, k block) space instead.  Costs are counted in k blocks per CTA; a last
//    lockstep round that runs part-empty costs less than its share suggests, because
//    full rounds are slowed by the L2 bandwidth all SMs draw together (measured: 0.30
//    us per k block for a lone CTA, 0.40 us with all 152 busy).
//  * M <= 128 (the probe's query rows): weight-bound.  Measured per-SM weight streams
//    through the TMA ring are ~29 / 55 / 65 GB/s for BN = 64 / 128 / 256, under an
//    aggregate of ~6.5 TB/s from HBM; a k split adds the last arriver's fixup, about
//    0.6 us per 32-column chunk and pair of partials, plus 1 us.
static GemmPlan plan_gemm(int M, int N, int K, EpiKind epi, int head_dim, bool w_kn = false) {
  const int sms = num_sms();
  const int tiles_m = (M + kBM - 1) / kBM;
  const int kb = K / kBK;
  auto valid = [&](int bn) {
    if (N % bn) return false;
    if (epi == EPI_SWIGLU && bn % 128) return false;
    if (epi == EPI_QKV_ROPE && bn % head_dim) return false;
    return true;
  };
  const int cands[3] = {256, 128, 64};
  if (tiles_m >= 2) {
    int bn = 64;
    for (int c : cands)
      if (valid(c)) {
        bn = c;
        break;
      }
    const int tiles = tiles_m * (N / bn);
    const long long lockstep = static_cast<long long>((tiles + sms - 1) / sms) * kb;
    const int groups = sms / tiles_m;
    const long long iters = static_cast<long long>(N / bn) * kb;
    if (groups >= 1 && tiles <= kCntCells && iters >= 4LL * groups && (iters + 1) * groups < (1LL << 31)) {
      const long long per = iters / groups;                                   // k blocks per CTA
      const long long parts = std::min<long long>(groups, (kb + per - 1) / per + 1);  // per shared tile, at most
      if (lockstep - per > kSkMinGain + kSkGainPerPart * std::max<long long>(0, parts - 2))
        return GemmPlan{bn, 1, tiles, groups};
    }
    // A residual add whose 256-wide tiles fill one lockstep round on part of the SMs
    // (the 832-row O projection: 112 tiles on 152 SMs) runs 224-wide tiles instead: more
    // CTAs, each with 7/8 of the work, the last column tile ragged.
    if (epi == EPI_ADD_F32 && !w_kn && bn == 256 && tiles <= sms) {
      const int tiles224 = tiles_m * ((N + 223) / 224);
      if (tiles224 > tiles && tiles224 <= sms) return GemmPlan{224, 1, tiles224, 0};
    }
    return GemmPlan{bn, 1, tiles, 0};
  }
  GemmPlan best{64, 1, tiles_m * (N / 64), 0};
  double best_t = 1e30;
  const double all_bytes = static_cast<double>(N) * K * 2.0;
  for (int bn : cands) {
    if (!valid(bn)) continue;
    const double stream = bn == 64 ? 29.0e9 : (bn == 128 ? 55.0e9 : 65.0e9);  // one SM's weight stream
    const int tiles = tiles_m * (N / bn);
    if (tiles > kCntCells) continue;
    for (int s = 1; s <= 8; ++s) {
      if (s > 1 && kb / s < 4) break;
      const int units = tiles * s;
      const int rounds = (units + sms - 1) / sms;
      const double unit_bytes = static_cast<double>(bn) * (static_cast<double>(K) / s) * 2.0;
      const double unit_flops = 2.0 * kBM * bn * (static_cast<double>(K) / s);
      double t = std::max(all_bytes / 6.5e12, rounds * std::max(unit_bytes / stream, unit_flops / 11.0e12));
      const double chunks = bn / 32.0;
      t += s > 1 ? 1.0e-6 + chunks * ((s + 1) / 2) * 0.6e-6 : chunks * 0.3e-6;
      if (t < best_t * 0.98) {
        best_t = t;
        best = GemmPlan{bn, s, tiles, 0};
      }
    }
  }
  return best;
}

// fp32 partial slots a plan writes (after the counters); 0 when no tile is shared
static size_t plan_part_bytes(const GemmPlan& p, int M) {
  const size_t slot = static_cast<size_t>(kBM) * p.BN * sizeof(float);
  if (p.groups > 0) {
    const int tiles_m = (M + kBM - 1) / kBM;
    return static_cast<size_t>(p.groups) * tiles_m * 2 * slot;
  }
  if (p.splits > 1) return static_cast<size_t>(p.tiles) * p.splits * slot;
  return 0;
}

size_t gemm_workspace_size(int M, int N, int K) {
  // the largest requirement over every epilogue's plan
  size_t need = 0;
  const EpiKind kinds[4] = {EPI_STORE_BF16, EPI_ADD_F32, EPI_QKV_ROPE, EPI_SWIGLU};
  for (EpiKind e : kinds) {
    for (int hd : {16, 64, 128}) {
      if (e != EPI_QKV_ROPE && hd != 16) continue;
      if (M <= 0 || N <= 0 || K <= 0 || N % 64 || K % 64) continue;
      const size_t b = plan_part_bytes(plan_gemm(M, N, K, e, hd), M);
      need = b > need ? b : need;
    }
  }
  return kCntBytes + need + 256;
}

qcf_status gemm_ws_prepare(void* ws, size_t ws_bytes, cudaStream_t st) {
  if (!ws || ws_bytes < kCntBytes) return set_error(QCF_ERR_WORKSPACE, "gemm: workspace %zu < %zu", ws_bytes, kCntBytes);
  const cudaError_t e = cudaMemsetAsync(ws, 0, kCntBytes, st);
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "gemm: counter reset");
}

template <int BN, int EPI, int HD, bool BMN = false>
static qcf_status launch_cfg(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tx, int M, int N,
                             int K, int splits, int groups, const EpiParams& ep, float* part, unsigned int* cnt,
                             cudaStream_t st, int grid, bool pdl) {
  using Cfg = GemmCfg<BN>;
  auto kern = gemm_tcgen05_kernel<BN, EPI, HD, BMN>;
  static PerDevice<cudaError_t> smem_attr;
  const cudaError_t attr_err = smem_attr.get(current_device(), [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return cuda_error(attr_err, "gemm: shared memory attribute");
  cudaError_t e = cudaSuccess;
  if (pdl) {
    e = launch_pdl(kern, dim3(grid), dim3(kGemmThreads), Cfg::SMEM_BYTES, st, ta, tb, tx, M, N, K, splits, groups, ep,
                   part, cnt, device_status_ptr());
  } else {
    kern<<<grid, kGemmThreads, Cfg::SMEM_BYTES, st>>>(ta, tb, tx, M, N, K, splits, groups, ep, part, cnt,
                                                       device_status_ptr());
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "gemm: launch");
}

template <int BN>
static qcf_status dispatch_kn(EpiKind epi, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tx, int M,
                              int N, int K,
                              int splits, int groups, const EpiParams& ep, float* part, unsigned int* cnt,
                              cudaStream_t st, int grid, bool pdl) {
  if constexpr (BN >= 64) {
    if (epi == EPI_STORE_BF16)
      return launch_cfg<BN, EPI_STORE_BF16, 0, true>(ta, tb, tx, M, N, K, splits, groups, ep, part, cnt, st, grid, pdl);
    if (epi == EPI_ADD_F32)
      return launch_cfg<BN, EPI_ADD_F32, 0, true>(ta, tb, tx, M, N, K, splits, groups, ep, part, cnt, st, grid, pdl);
  }
  return set_error(QCF_ERR_UNSUPPORTED, "gemm: [K][N] weights support the store and add epilogues only");
}

template <int BN>
static qcf_status dispatch_epi(EpiKind epi, int hd, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tx,
                               int M, int N, int K,
                               int splits, int groups, const EpiParams& ep, float* part, unsigned int* cnt,
                               cudaStream_t st, int grid, bool pdl) {
  switch (epi) {
    case EPI_STORE_BF16: return launch_cfg<BN, EPI_STORE_BF16, 0, false>(ta, tb, tx, M, N, K, splits, groups, ep, part, cnt, st, grid, pdl);
    case EPI_ADD_F32: return launch_cfg<BN, EPI_ADD_F32, 0, false>(ta, tb, tx, M, N, K, splits, groups, ep, part, cnt, st, grid, pdl);
    case EPI_SWIGLU:
      if constexpr (BN >= 128) return launch_cfg<BN, EPI_SWIGLU, 0, false>(ta, tb, tx, M, N, K, splits, groups, ep, part, cnt, st, grid, pdl);
      break;
    case EPI_QKV_ROPE:
      if (hd == 16) return launch_cfg<BN, EPI_QKV_ROPE, 16, false>(ta, tb, tx, M, N, K, splits, groups, ep, part, cnt, st, grid, pdl);
      if (hd == 64) return launch_cfg<BN, EPI_QKV_ROPE, 64, false>(ta, tb, tx, M, N, K, splits, groups, ep, part, cnt, st, grid, pdl);
      if constexpr (BN >= 128)
        if (hd == 128) return launch_cfg<BN, EPI_QKV_ROPE, 128, false>(ta, tb, tx, M, N, K, splits, groups, ep, part, cnt, st, grid, pdl);
      break;
  }
  return set_error(QCF_ERR_UNSUPPORTED, "gemm: no kernel for epilogue %d, BN %d, head dim %d", epi, BN, hd);
}

qcf_status gemm_launch(EpiKind epi, const __nv_bfloat16* A, int M, int K, const __nv_bfloat16* W, int N,
                       const EpiParams& ep, void* ws, size_t ws_bytes, cudaStream_t st, KernelClass kc, bool w_kn,
                       bool pdl, bool ws_zeroed) {
  if (M <= 0) return QCF_OK;
  if (K % kBK || N % 64 || K <= 0 || N <= 0) return set_error(QCF_ERR_SHAPE, "gemm: K=%d N=%d (K%%64, N%%64 required)", K, N);
  const int hd = epi == EPI_QKV_ROPE ? ep.D : 16;
  GemmPlan p = plan_gemm(M, N, K, epi, hd, w_kn);
  float* part = nullptr;
  unsigned int* cnt = nullptr;
  if (p.splits > 1 || p.groups > 0) {
    const size_t need = kCntBytes + plan_part_bytes(p, M);
    if (!ws || ws_bytes < need) return set_error(QCF_ERR_WORKSPACE, "gemm: workspace %zu < %zu", ws_bytes, need);
    cnt = static_cast<unsigned int*>(ws);
    part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCntBytes);
    if (!ws_zeroed) {
      const cudaError_t e = cudaMemsetAsync(cnt, 0, p.tiles * sizeof(unsigned int), st);
      if (e != cudaSuccess) return cuda_error(e, "gemm: counter reset");
    }
  }
  CUtensorMap ta, tb, tx;
  // the residual-add epilogue stages x through TMA boxes of 32 rows x 32 fp32
  const bool tx_ok = epi != EPI_ADD_F32 ||
                     encode_tmap_2d(&tx, ep.out, N, M, static_cast<uint64_t>(ep.ldo) * 4, 32, 32,
                                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
  const bool tb_ok = w_kn ? encode_tmap_2d(&tb, W, N, K, static_cast<uint64_t>(N) * 2, 64, kBK, CU_TENSOR_MAP_SWIZZLE_128B)
                          : encode_tmap_2d(&tb, W, K, N, static_cast<uint64_t>(K) * 2, kBK, p.BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!encode_tmap_2d(&ta, A, K, M, static_cast<uint64_t>(K) * 2, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tb_ok || !tx_ok)
    return set_error(QCF_ERR_CUDA, "gemm: tensor map encoding failed");
  if (epi != EPI_ADD_F32) tx = ta;  // unused by the other epilogues
  const int units = p.tiles * p.splits;
  const int grid = p.groups > 0 ? p.groups * ((M + kBM - 1) / kBM) : (units < num_sms() ? units : num_sms());
  LaunchScope ls(kc, st);
  if (w_kn) {
    switch (p.BN) {
      case 256: return dispatch_kn<256>(epi, ta, tb, tx, M, N, K, p.splits, p.groups, ep, part, cnt, st, grid, pdl);
      case 128: return dispatch_kn<128>(epi, ta, tb, tx, M, N, K, p.splits, p.groups, ep, part, cnt, st, grid, pdl);
      default: return dispatch_kn<64>(epi, ta, tb, tx, M, N, K, p.splits, p.groups, ep, part, cnt, st, grid, pdl);
    }
  }
  switch (p.BN) {
    case 224:  // residual add only (plan_gemm)
      if (epi != EPI_ADD_F32) return set_error(QCF_ERR_UNSUPPORTED, "gemm: BN 224 serves the residual add only");
      return launch_cfg<224, EPI_ADD_F32, 0, false>(ta, tb, tx, M, N, K, p.splits, p.groups, ep, part, cnt, st, grid, pdl);
    case 256: return dispatch_epi<256>(epi, hd, ta, tb, tx, M, N, K, p.splits, p.groups, ep, part, cnt, st, grid, pdl);
    case 128: return dispatch_epi<128>(epi, hd, ta, tb, tx, M, N, K, p.splits, p.groups, ep, part, cnt, st, grid, pdl);
    default: return dispatch_epi<64>(epi, hd, ta, tb, tx, M, N, K, p.splits, p.groups, ep, part, cnt, st, grid, pdl);
  }
}

}  // namespace qcf

using namespace qcf;

extern "C" {

size_t qcf_linear_workspace_size(int M, int N, int K) { return gemm_workspace_size(M, N, K); }

qcf_status qcf_linear(const qcf_bf16* A, int M, int K, const qcf_bf16* W, int N, int epilogue, void* out, void* ws,
                      size_t ws_bytes, void* stream) {
  if (!A || !W || !out) return set_error(QCF_ERR_INVALID_ARG, "qcf_linear: NULL pointer");
  const bool w_kn = (epilogue & QCF_LINEAR_W_KN) != 0;
  epilogue &= ~QCF_LINEAR_W_KN;
  if (epilogue != QCF_EPI_STORE_BF16 && epilogue != QCF_EPI_ADD_F32)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_linear: unknown epilogue %d", epilogue);
  if (M < 0 || K <= 0 || N <= 0 || K % 64 || N % 64)
    return set_error(QCF_ERR_SHAPE, "qcf_linear: M=%d K=%d N=%d (K, N multiples of 64)", M, K, N);
  if (take_fault(4) || !aligned16(A) || !aligned16(W) || !aligned16(out))
    return set_error(QCF_ERR_ALIGN, "qcf_linear: pointers must be 16-byte aligned");
  if (take_fault(2)) return set_error(QCF_ERR_WORKSPACE, "qcf_linear: injected short workspace");
  EpiParams ep{};
  ep.out = out;
  ep.ldo = N;
  return gemm_launch(epilogue == QCF_EPI_STORE_BF16 ? EPI_STORE_BF16 : EPI_ADD_F32,
                     reinterpret_cast<const __nv_bfloat16*>(A), M, K, reinterpret_cast<const __nv_bfloat16*>(W), N, ep,
                     ws, ws_bytes, static_cast<cudaStream_t>(stream), KC_GEMM_OTHER, w_kn);
}

}  // extern "C"
