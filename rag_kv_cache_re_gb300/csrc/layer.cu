// Decoder layer forward for recomputed rows, full prefill, and the per-request
// fused-prefill driver (probe -> profile -> top-N -> pipelined per-layer recompute).
#include <errno.h>
#include <fcntl.h>
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <condition_variable>
#include <functional>
#include <map>
#include <thread>
#include <mutex>
#include <tuple>
#include <vector>

#include "qcf_internal.cuh"

namespace qcf {

// ------------------------------------------------------------------ workspace carving

struct Carve {
  uint8_t* base;
  size_t cap;
  size_t used = 0;
  bool ok = true;
  template <typename T>
  T* take(size_t count) {
    const size_t off = align_up(used, 256);
    const size_t bytes = align_up(count * sizeof(T), 256);
    used = off + bytes;
    if (!base || used > cap) {
      ok = false;
      return nullptr;
    }
    return reinterpret_cast<T*>(base + off);
  }
};

static size_t gemm_ws_layer(const qcf_dims& d, int n) {
  const int D = d.head_dim;
  size_t w = gemm_workspace_size(n, (d.n_heads + 2 * d.n_kv_heads) * D, d.d_model);
  w = std::max(w, gemm_workspace_size(n, d.d_model, d.n_heads * D));
  w = std::max(w, gemm_workspace_size(n, 2 * d.ffn_padded, d.d_model));
  w = std::max(w, gemm_workspace_size(n, d.d_model, d.ffn_padded));
  return w;
}

struct LayerBufs {
  __nv_bfloat16* h;
  __nv_bfloat16* q;
  __nv_bfloat16* o;
  __nv_bfloat16* act;
  void* gemm_ws;
  size_t gemm_ws_bytes;
  bool gemm_zeroed = false;  // its GEMM counters were zeroed on the stream the GEMMs run on
  void* attn_ws;
  size_t attn_ws_bytes;
};

static size_t layer_ws_bytes(const qcf_dims& d, int n, int T) {
  Carve c{nullptr, 0};
  c.take<__nv_bfloat16>(static_cast<size_t>(n) * d.d_model);
  c.take<__nv_bfloat16>(static_cast<size_t>(n) * d.n_heads * d.head_dim);
  c.take<__nv_bfloat16>(static_cast<size_t>(n) * d.n_heads * d.head_dim);
  c.take<__nv_bfloat16>(static_cast<size_t>(n) * d.ffn_padded);
  c.take<uint8_t>(gemm_ws_layer(d, n));
  c.take<uint8_t>(attn_workspace_size(n, T, d.n_heads, d.n_kv_heads, d.head_dim));
  return c.used;
}

static bool carve_layer(Carve& c, const qcf_dims& d, int n, int T, LayerBufs* b) {
  b->h = c.take<__nv_bfloat16>(static_cast<size_t>(n) * d.d_model);
  b->q = c.take<__nv_bfloat16>(static_cast<size_t>(n) * d.n_heads * d.head_dim);
  b->o = c.take<__nv_bfloat16>(static_cast<size_t>(n) * d.n_heads * d.head_dim);
  b->act = c.take<__nv_bfloat16>(static_cast<size_t>(n) * d.ffn_padded);
  b->gemm_ws_bytes = gemm_ws_layer(d, n);
  b->gemm_ws = c.take<uint8_t>(b->gemm_ws_bytes);
  b->attn_ws_bytes = attn_workspace_size(n, T, d.n_heads, d.n_kv_heads, d.head_dim);
  b->attn_ws = c.take<uint8_t>(b->attn_ws_bytes);
  return c.ok;
}

static qcf_status check_dims(const qcf_dims& d, const char* who) {
  const int D = d.head_dim;
  if (d.n_layers <= 0 || d.d_model <= 0 || d.n_heads <= 0 || d.n_kv_heads <= 0 || d.n_heads % d.n_kv_heads ||
      d.n_heads / d.n_kv_heads > 8 || (D != 16 && D != 64 && D != 128) || d.d_model % 64 || (d.n_heads * D) % 64 ||
      d.ffn <= 0 || d.ffn_padded < d.ffn || d.ffn_padded % 64 || d.vocab <= 0 || d.d_model > 8192)
    return set_error(QCF_ERR_SHAPE,
                     "%s: unsupported dims (L=%d d=%d Hq=%d Hkv=%d D=%d ffn=%d ffn_padded=%d vocab=%d); need D in "
                     "{16,64,128}, d%%64==0, Hq*D%%64==0, ffn_padded%%64==0, Hq/Hkv<=8",
                     who, d.n_layers, d.d_model, d.n_heads, d.n_kv_heads, D, d.ffn, d.ffn_padded, d.vocab);
  return QCF_OK;
}

static qcf_status check_model(const qcf_model* m, const char* who) {
  if (!m || !m->layers || !m->embed || !m->lm_head || !m->g_final || !m->rope.cos || !m->rope.sin)
    return set_error(QCF_ERR_INVALID_ARG, "%s: model has NULL pointers", who);
  qcf_status s = check_dims(m->dims, who);
  if (s != QCF_OK) return s;
  if (m->rope.head_dim != m->dims.head_dim) return set_error(QCF_ERR_SHAPE, "%s: RoPE table head dim mismatch", who);
  return QCF_OK;
}

// One decoder layer on rows x (validated by the caller).
// `probe` only selects the timing classes (the probe's 64-row GEMMs are weight-bound
// and are accounted apart from the recompute GEMMs).
// The first kernel is launched plainly unless the caller knows it follows this
// library's kernels directly (first_pdl); for layers of up to kPdlMaxRows rows the six
// after it, which follow this
// library's kernels directly, are launched programmatically so each one's set-up
// overlaps the tail of the one before.  Measured on GB300 (8B layer shapes): the
// 64- and 832-row layers of a fused prefill gain ~5% per request; the 5184-row layers
// of a full prefill lose ~1.5% (their kernels run several waves and the next kernel's
// parked CTAs gain nothing there), so those stay plain.
constexpr int kPdlMaxRows = 2048;
static qcf_status layer_forward_impl(const qcf_model* m, int layer, float* x, const int32_t* rope_pos,
                                     const int32_t* cache_row, int n, __nv_bfloat16* Kc, __nv_bfloat16* Vc, int T,
                                     const LayerBufs& b, cudaStream_t st, bool probe = false,
                                     bool first_pdl = false, const int32_t* key0 = nullptr) {
  const qcf_dims& d = m->dims;
  const qcf_layer_weights& w = m->layers[layer];
  const int D = d.head_dim, Hq = d.n_heads, Hkv = d.n_kv_heads;
  const bool pdl = n <= kPdlMaxRows;
  cudaError_t e = launch_rmsnorm(x, n, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.g_attn), d.eps, b.h, st,
                                 first_pdl && pdl);
  if (e != cudaSuccess) return cuda_error(e, "layer: rmsnorm");
  EpiParams ep{};
  ep.q_out = b.q;
  ep.k_cache = Kc;
  ep.v_cache = Vc;
  ep.rope_pos = rope_pos;
  ep.cache_row = cache_row;
  ep.cos_t = m->rope.cos;
  ep.sin_t = m->rope.sin;
  ep.Hq = Hq;
  ep.Hkv = Hkv;
  ep.D = D;
  ep.T = T;
  ep.max_pos = m->rope.max_pos;
  ep.status = device_status_ptr();
  qcf_status s = gemm_launch(EPI_QKV_ROPE, b.h, n, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.w_qkv),
                             (Hq + 2 * Hkv) * D, ep, b.gemm_ws, b.gemm_ws_bytes, st, probe ? KC_GEMM_PROBE : KC_GEMM_QKV,
                             false, pdl, b.gemm_zeroed);
  if (s != QCF_OK) return s;
  s = attn_launch(b.q, cache_row, n, Kc, Vc, T, Hq, Hkv, D, 1.0f / sqrtf(static_cast<float>(D)), b.o, nullptr, b.attn_ws,
                  b.attn_ws_bytes, st, probe ? KC_ATTN_PROBE : KC_ATTN, pdl, key0);
  if (s != QCF_OK) return s;
  EpiParams eo{};
  eo.out = x;
  eo.ldo = d.d_model;
  s = gemm_launch(EPI_ADD_F32, b.o, n, Hq * D, reinterpret_cast<const __nv_bfloat16*>(w.w_o), d.d_model, eo, b.gemm_ws,
                  b.gemm_ws_bytes, st, probe ? KC_GEMM_PROBE : KC_GEMM_O, false, pdl, b.gemm_zeroed);
  if (s != QCF_OK) return s;
  e = launch_rmsnorm(x, n, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.g_mlp), d.eps, b.h, st, pdl);
  if (e != cudaSuccess) return cuda_error(e, "layer: rmsnorm");
  EpiParams eg{};
  eg.out = b.act;
  eg.ldo = d.ffn_padded;
  s = gemm_launch(EPI_SWIGLU, b.h, n, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.w_gu), 2 * d.ffn_padded, eg,
                  b.gemm_ws, b.gemm_ws_bytes, st, probe ? KC_GEMM_PROBE : KC_GEMM_GU, false, pdl, b.gemm_zeroed);
  if (s != QCF_OK) return s;
  EpiParams edn{};
  edn.out = x;
  edn.ldo = d.d_model;
  return gemm_launch(EPI_ADD_F32, b.act, n, d.ffn_padded, reinterpret_cast<const __nv_bfloat16*>(w.w_down), d.d_model,
                     edn, b.gemm_ws, b.gemm_ws_bytes, st, probe ? KC_GEMM_PROBE : KC_GEMM_DOWN, false, pdl, b.gemm_zeroed);
}

// ------------------------------------------------------------------ small helper kernels

// out[i] = start + i
__global__ void iota_kernel(int32_t* out, int n, int start) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = start + i;
}

// rows[i] = sel[i] for i < N, then the query rows C, C+1, ...
__global__ void make_rows_kernel(const int32_t* __restrict__ sel, int N, int C, int n, int32_t* __restrict__ rows) {
  pdl_wait();  // the selection comes from the kernel before
  pdl_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) rows[i] = i < N ? sel[i] : C + (i - N);
}

// HKVD compaction: keep_idx[i] = sel_idx[i] for i < N (context rows kept, indices into
// the previous row list), then the query rows, which follow the n_ctx context rows
// there; rows_new[i] = rows_prev[keep_idx[i]].
__global__ void keep_rows_kernel(const int32_t* __restrict__ sel_idx, int N, int n_ctx, int n,
                                 const int32_t* __restrict__ rows_prev, int32_t* __restrict__ keep_idx,
                                 int32_t* __restrict__ rows_new) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int k = i < N ? sel_idx[i] : n_ctx + (i - N);
  keep_idx[i] = k;
  rows_new[i] = rows_prev[k];
}

// dst[i] += src[i]
__global__ void add_f32_kernel(float* __restrict__ dst, const float* __restrict__ src, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] += src[i];
}

constexpr int kMaxReqChunks = 512;
struct ChunkOffsets {
  int n_chunks;
  int off[kMaxReqChunks];
};

// Probe KV prefix for one layer: anchor rows of every chunk from the staging
// buffer [chunk][layer][anchor][Hkv*D] into probe cache rows chunk*A + a of every
// probe layer (layer l's cache at l * layer_stride elements), keys re-rotated by the
// chunk's offset, values copied.  One thread per (layer, row, head, group of 8
// rotation pairs).
__global__ void anchor_assemble_kernel(const __nv_bfloat16* __restrict__ stK, const __nv_bfloat16* __restrict__ stV,
                                       int n_layers_staged, int A, int Hkv, int D,
                                       const float* __restrict__ cos_t, const float* __restrict__ sin_t,
                                       const ChunkOffsets co, __nv_bfloat16* __restrict__ pK,
                                       __nv_bfloat16* __restrict__ pV, size_t layer_stride) {
  const int half = D / 2, groups = half / 8;
  const int per_row = Hkv * groups;
  const int rows = co.n_chunks * A;
  const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gtid >= static_cast<long long>(n_layers_staged) * rows * per_row) return;
  const int layer = static_cast<int>(gtid / (static_cast<long long>(rows) * per_row));
  const int tid = static_cast<int>(gtid - static_cast<long long>(layer) * rows * per_row);
  pK += static_cast<size_t>(layer) * layer_stride;
  pV += static_cast<size_t>(layer) * layer_stride;
  const int row = tid / per_row;
  const int rem = tid - row * per_row;
  const int h = rem / groups, k0 = (rem - h * groups) * 8;
  const int c = row / A, a = row - c * A;
  const size_t HD = static_cast<size_t>(Hkv) * D;
  const size_t src = ((static_cast<size_t>(c) * n_layers_staged + layer) * A + a) * HD + static_cast<size_t>(h) * D;
  const size_t dst = static_cast<size_t>(row) * HD + static_cast<size_t>(h) * D;
  const int delta = co.off[c];
  const __nv_bfloat162* ka = reinterpret_cast<const __nv_bfloat162*>(stK + src + k0);
  const __nv_bfloat162* kb = reinterpret_cast<const __nv_bfloat162*>(stK + src + half + k0);
  const float* cs = cos_t + static_cast<size_t>(delta) * half + k0;
  const float* sn = sin_t + static_cast<size_t>(delta) * half + k0;
  __nv_bfloat162 o1[4], o2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 av = __bfloat1622float2(ka[i]), bv = __bfloat1622float2(kb[i]);
    o1[i] = __floats2bfloat162_rn(av.x * cs[2 * i] - bv.x * sn[2 * i], av.y * cs[2 * i + 1] - bv.y * sn[2 * i + 1]);
    o2[i] = __floats2bfloat162_rn(bv.x * cs[2 * i] + av.x * sn[2 * i], bv.y * cs[2 * i + 1] + av.y * sn[2 * i + 1]);
  }
  *reinterpret_cast<uint4*>(pK + dst + k0) = *reinterpret_cast<uint4*>(o1);
  *reinterpret_cast<uint4*>(pK + dst + half + k0) = *reinterpret_cast<uint4*>(o2);
  *reinterpret_cast<uint4*>(pV + dst + k0) = *reinterpret_cast<const uint4*>(stV + src + k0);
  *reinterpret_cast<uint4*>(pV + dst + half + k0) = *reinterpret_cast<const uint4*>(stV + src + half + k0);
}

// ------------------------------------------------------------------ request plan

struct RequestLayout {
  int C, Q, T, N, ns, nA, crit;
  LayerBufs lb;          // sized for max(ns rows over T, Q rows over nA+Q)
  float* x;              // [ns][d]
  int32_t* rows;         // [ns]
  int32_t* probe_pos;    // [Q] absolute positions C..T-1
  int32_t* probe_row;    // [Q] probe cache rows nA..nA+Q-1
  __nv_bfloat16* stK;    // [n_chunks][crit][A][HD]
  __nv_bfloat16* stV;
  __nv_bfloat16* pK;     // [crit][nA+Q][HD]: the probe cache of each probe layer
  __nv_bfloat16* pV;
  __nv_bfloat16* q_crit; // [Q][Hq*D]
  float* scores;         // [C]
  float* scores_acc;     // [C] QCAll: the probe layers' scores
  float* scores_tmp;     // [C] QCAll: one layer's scores
  int32_t* sel;          // [N]
  void* prof_ws;
  size_t prof_ws_bytes;
  void* lm_ws;
  void* topn_ws;         // the cooperative top-N's scratch (context above 16384 tokens)
  size_t topn_ws_bytes;
};

static bool carve_request(Carve& c, const qcf_dims& d, int C, int Q, int nA, int N, int n_chunks, int crit,
                          int n_anchor, RequestLayout* r) {
  const int T = C + Q, ns = N + Q;
  const size_t HD = static_cast<size_t>(d.n_kv_heads) * d.head_dim;
  r->C = C; r->Q = Q; r->T = T; r->N = N; r->ns = ns; r->nA = nA; r->crit = crit;
  const int nmax = ns > Q ? ns : Q;
  r->lb.h = c.take<__nv_bfloat16>(static_cast<size_t>(nmax) * d.d_model);
  r->lb.q = c.take<__nv_bfloat16>(static_cast<size_t>(nmax) * d.n_heads * d.head_dim);
  r->lb.o = c.take<__nv_bfloat16>(static_cast<size_t>(nmax) * d.n_heads * d.head_dim);
  r->lb.act = c.take<__nv_bfloat16>(static_cast<size_t>(nmax) * d.ffn_padded);
  r->lb.gemm_ws_bytes = std::max(gemm_ws_layer(d, ns), gemm_ws_layer(d, Q));
  r->lb.gemm_ws = c.take<uint8_t>(r->lb.gemm_ws_bytes);
  r->lb.attn_ws_bytes = std::max(attn_workspace_size(ns, T, d.n_heads, d.n_kv_heads, d.head_dim),
                                 attn_workspace_size(Q, nA + Q, d.n_heads, d.n_kv_heads, d.head_dim));
  r->lb.attn_ws = c.take<uint8_t>(r->lb.attn_ws_bytes);
  r->x = c.take<float>(static_cast<size_t>(nmax) * d.d_model);
  r->rows = c.take<int32_t>(ns);
  r->probe_pos = c.take<int32_t>(Q);
  r->probe_row = c.take<int32_t>(Q);
  const size_t staged = static_cast<size_t>(n_chunks) * (crit > 0 ? crit : 1) * (n_anchor > 0 ? n_anchor : 1) * HD;
  r->stK = c.take<__nv_bfloat16>(staged);
  r->stV = c.take<__nv_bfloat16>(staged);
  // one probe cache per probe layer, so every layer's anchor rows are assembled in one launch
  const size_t probe_layers = crit > 0 ? crit : 1;
  r->pK = c.take<__nv_bfloat16>(probe_layers * (nA + Q) * HD);
  r->pV = c.take<__nv_bfloat16>(probe_layers * (nA + Q) * HD);
  r->q_crit = c.take<__nv_bfloat16>(static_cast<size_t>(Q) * d.n_heads * d.head_dim);
  r->scores = c.take<float>(C);
  r->scores_acc = c.take<float>(C);
  r->scores_tmp = c.take<float>(C);
  r->sel = c.take<int32_t>(N > 0 ? N : 1);
  r->topn_ws_bytes = qcf_topn_select_workspace_size(C);   // 0 up to 16384 context tokens
  r->topn_ws = c.take<uint8_t>(r->topn_ws_bytes > 0 ? r->topn_ws_bytes : 1);
  r->prof_ws_bytes = qcf_profile_scores_workspace_size(Q, C, d.n_heads, d.n_kv_heads, d.head_dim);
  r->prof_ws = c.take<uint8_t>(r->prof_ws_bytes);
  r->lm_ws = c.take<uint8_t>(qcf_lm_head_workspace_size(&d));
  return c.ok;
}

// ------------------------------------------------------------------ HKVD (CacheBlend) selection

// Buffers of the KV-deviation path.  Layer 0 projects K/V for all T rows, so the
// projection buffers hold T rows; the kept rows (at most N_0 + Q) get the rest.
struct HkvdLayout {
  int C, Q, T, N0, nk;    // nk = N_0 + Q
  float* x_a;             // [T][d]   rows of the previous layer / kept rows, alternating
  float* x_b;             // [T][d]
  int32_t* rows_a;        // [T] positions
  int32_t* rows_b;        // [T]
  int32_t* iota;          // [T] 0..T-1: temporary K/V rows of the projection
  __nv_bfloat16* h;       // [T][d]
  __nv_bfloat16* q;       // [T][Hq*D]
  __nv_bfloat16* k_tmp;   // [T][HD]
  __nv_bfloat16* v_tmp;   // [T][HD]
  __nv_bfloat16* q_keep;  // [nk][Hq*D]
  __nv_bfloat16* k_keep;  // [nk][HD]
  __nv_bfloat16* v_keep;  // [nk][HD]
  float* dev;             // [C]
  int32_t* sel_idx;       // [max(N_0, 1)]
  int32_t* keep_idx;      // [nk]
  LayerBufs lb;           // o, act and the GEMM / attention workspaces for nk rows (h, q unused)
  void* lm_ws;
};

static bool hkvd_counts(const int32_t* sched, int L, int C, int ratio_bp, std::vector<int>* Nl) {
  if (!sched) return false;
  Nl->assign(L, 0);
  for (int l = 0; l < L; ++l) {
    if (sched[l] < 0 || sched[l] > 10000 || (l > 0 && sched[l] > sched[l - 1])) return false;
    qcf_num_selected(C, sched[l], &(*Nl)[l]);
  }
  return sched[L - 1] == ratio_bp;
}

static bool carve_hkvd(Carve& c, const qcf_dims& d, int C, int Q, const std::vector<int>& Nl, HkvdLayout* H) {
  const int T = C + Q, N0 = Nl.empty() ? 0 : Nl[0], nk = N0 + Q;
  const size_t HD = static_cast<size_t>(d.n_kv_heads) * d.head_dim, QD = static_cast<size_t>(d.n_heads) * d.head_dim;
  H->C = C; H->Q = Q; H->T = T; H->N0 = N0; H->nk = nk;
  H->x_a = c.take<float>(static_cast<size_t>(T) * d.d_model);
  H->x_b = c.take<float>(static_cast<size_t>(T) * d.d_model);
  H->rows_a = c.take<int32_t>(T);
  H->rows_b = c.take<int32_t>(T);
  H->iota = c.take<int32_t>(T);
  H->h = c.take<__nv_bfloat16>(static_cast<size_t>(T) * d.d_model);
  H->q = c.take<__nv_bfloat16>(static_cast<size_t>(T) * QD);
  H->k_tmp = c.take<__nv_bfloat16>(static_cast<size_t>(T) * HD);
  H->v_tmp = c.take<__nv_bfloat16>(static_cast<size_t>(T) * HD);
  H->q_keep = c.take<__nv_bfloat16>(static_cast<size_t>(nk) * QD);
  H->k_keep = c.take<__nv_bfloat16>(static_cast<size_t>(nk) * HD);
  H->v_keep = c.take<__nv_bfloat16>(static_cast<size_t>(nk) * HD);
  H->dev = c.take<float>(C > 0 ? C : 1);
  H->sel_idx = c.take<int32_t>(N0 > 0 ? N0 : 1);
  H->keep_idx = c.take<int32_t>(nk);
  H->lb.h = H->h;
  H->lb.q = H->q_keep;
  H->lb.o = c.take<__nv_bfloat16>(static_cast<size_t>(nk) * QD);
  H->lb.act = c.take<__nv_bfloat16>(static_cast<size_t>(nk) * d.ffn_padded);
  size_t gws = std::max(gemm_ws_layer(d, T), gemm_ws_layer(d, nk));
  size_t aws = 0;
  for (int l = 0; l < static_cast<int>(Nl.size()); ++l) {
    gws = std::max(gws, gemm_ws_layer(d, Nl[l] + Q));
    aws = std::max(aws, attn_workspace_size(Nl[l] + Q, T, d.n_heads, d.n_kv_heads, d.head_dim));
  }
  H->lb.gemm_ws_bytes = gws;
  H->lb.gemm_ws = c.take<uint8_t>(gws);
  H->lb.attn_ws_bytes = aws;
  H->lb.attn_ws = c.take<uint8_t>(aws > 0 ? aws : 1);
  H->lm_ws = c.take<uint8_t>(qcf_lm_head_workspace_size(&d));
  return c.ok;
}

// One layer of the KV-deviation path.  In: x_prev [n_prev][d] at positions rows_prev
// (the n_ctx context rows kept so far, then the Q query rows).  Projects K/V for all
// of them, measures the context rows' deviation against the layer's reused cache,
// keeps the top N of those, compacts the kept rows plus the query into x_new /
// rows_new, writes their fresh K/V into the cache and runs attention, O and the MLP
// for them.  dev0 (layer 0 only, nullable) receives the deviations.
static qcf_status hkvd_layer(const qcf_model* m, int l, HkvdLayout& H, const float* x_prev, const int32_t* rows_prev,
                             int n_ctx, int N, float* x_new, int32_t* rows_new, __nv_bfloat16* Kl, __nv_bfloat16* Vl,
                             float* dev_out, int32_t* sel_out, cudaStream_t st) {
  const qcf_dims& d = m->dims;
  const qcf_layer_weights& w = m->layers[l];
  const int D = d.head_dim, Hq = d.n_heads, Hkv = d.n_kv_heads, Q = H.Q, T = H.T;
  const int n_prev = n_ctx + Q, nk = N + Q;
  const int HD = Hkv * D, QD = Hq * D;
  cudaError_t e = launch_rmsnorm(x_prev, n_prev, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.g_attn), d.eps, H.h, st);
  if (e != cudaSuccess) return cuda_error(e, "hkvd: rmsnorm");
  EpiParams ep{};
  ep.q_out = H.q;
  ep.k_cache = H.k_tmp;
  ep.v_cache = H.v_tmp;
  ep.rope_pos = rows_prev;
  ep.cache_row = H.iota;
  ep.cos_t = m->rope.cos;
  ep.sin_t = m->rope.sin;
  ep.Hq = Hq;
  ep.Hkv = Hkv;
  ep.D = D;
  ep.T = n_prev;
  ep.max_pos = m->rope.max_pos;
  ep.status = device_status_ptr();
  qcf_status s = gemm_launch(EPI_QKV_ROPE, H.h, n_prev, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.w_qkv),
                             (Hq + 2 * Hkv) * D, ep, H.lb.gemm_ws, H.lb.gemm_ws_bytes, st, KC_GEMM_QKV, false, false,
                             H.lb.gemm_zeroed);
  if (s != QCF_OK) return s;
  float* dev = dev_out ? dev_out : H.dev;
  if ((e = launch_kv_deviation(H.k_tmp, H.v_tmp, rows_prev, n_ctx, Kl, Vl, T, HD, dev, st)) != cudaSuccess)
    return cuda_error(e, "hkvd: deviation");
  if (N > 0 && (s = qcf_topn_select(dev, n_ctx, N, H.sel_idx, st)) != QCF_OK) return s;
  {
    LaunchScope ls(KC_MISC, st);
    keep_rows_kernel<<<(nk + 255) / 256, 256, 0, st>>>(H.sel_idx, N, n_ctx, nk, rows_prev, H.keep_idx, rows_new);
  }
  // compact: hidden rows (fp32, moved as 2d bf16-sized words), q and the fresh K/V
  if ((s = qcf_gather_rows(reinterpret_cast<const qcf_bf16*>(x_prev), n_prev, 2 * d.d_model, H.keep_idx, nk,
                           reinterpret_cast<qcf_bf16*>(x_new), st)) != QCF_OK ||
      (s = qcf_gather_rows(reinterpret_cast<const qcf_bf16*>(H.q), n_prev, QD, H.keep_idx, nk,
                           reinterpret_cast<qcf_bf16*>(H.q_keep), st)) != QCF_OK ||
      (s = qcf_gather_rows(reinterpret_cast<const qcf_bf16*>(H.k_tmp), n_prev, HD, H.keep_idx, nk,
                           reinterpret_cast<qcf_bf16*>(H.k_keep), st)) != QCF_OK ||
      (s = qcf_gather_rows(reinterpret_cast<const qcf_bf16*>(H.v_tmp), n_prev, HD, H.keep_idx, nk,
                           reinterpret_cast<qcf_bf16*>(H.v_keep), st)) != QCF_OK)
    return s;
  if ((s = qcf_scatter_kv(reinterpret_cast<const qcf_bf16*>(H.k_keep), reinterpret_cast<const qcf_bf16*>(H.v_keep),
                          rows_new, nk, Hkv, D, reinterpret_cast<qcf_bf16*>(Kl), reinterpret_cast<qcf_bf16*>(Vl), T,
                          st)) != QCF_OK)
    return s;
  if (sel_out && N > 0 &&
      (e = cudaMemcpyAsync(sel_out, rows_new, N * sizeof(int32_t), cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
    return cuda_error(e, "hkvd: selection copy");
  // attention, O projection and the MLP for the kept rows
  s = attn_launch(H.q_keep, rows_new, nk, Kl, Vl, T, Hq, Hkv, D, 1.0f / sqrtf(static_cast<float>(D)), H.lb.o, nullptr,
                  H.lb.attn_ws, H.lb.attn_ws_bytes, st, KC_ATTN);
  if (s != QCF_OK) return s;
  EpiParams eo{};
  eo.out = x_new;
  eo.ldo = d.d_model;
  s = gemm_launch(EPI_ADD_F32, H.lb.o, nk, QD, reinterpret_cast<const __nv_bfloat16*>(w.w_o), d.d_model, eo,
                  H.lb.gemm_ws, H.lb.gemm_ws_bytes, st, KC_GEMM_O, false, false, H.lb.gemm_zeroed);
  if (s != QCF_OK) return s;
  if ((e = launch_rmsnorm(x_new, nk, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.g_mlp), d.eps, H.h, st)) !=
      cudaSuccess)
    return cuda_error(e, "hkvd: rmsnorm");
  EpiParams eg{};
  eg.out = H.lb.act;
  eg.ldo = d.ffn_padded;
  s = gemm_launch(EPI_SWIGLU, H.h, nk, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.w_gu), 2 * d.ffn_padded, eg,
                  H.lb.gemm_ws, H.lb.gemm_ws_bytes, st, KC_GEMM_GU, false, false, H.lb.gemm_zeroed);
  if (s != QCF_OK) return s;
  EpiParams edn{};
  edn.out = x_new;
  edn.ldo = d.d_model;
  return gemm_launch(EPI_ADD_F32, H.lb.act, nk, d.ffn_padded, reinterpret_cast<const __nv_bfloat16*>(w.w_down),
                     d.d_model, edn, H.lb.gemm_ws, H.lb.gemm_ws_bytes, st, KC_GEMM_DOWN, false, false, H.lb.gemm_zeroed);
}

struct EventPool {
  std::mutex mu;
  std::vector<cudaEvent_t> ev;
  bool get(size_t n, cudaEvent_t** out) {
    while (ev.size() < n) {
      cudaEvent_t e;
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
      ev.push_back(e);
    }
    *out = ev.data();
    return true;
  }
};
static EventPool& event_pool() {
  static EventPool p;
  return p;
}

// Everything a request needs between validation and its launches.
// Pinned host memory feeds a layer's chunk K/V (~10 MB for the 8B request) faster
// than a 832-row layer recomputes, so the copies run several layers ahead: the
// recompute waits for them every 4 layers.
constexpr int kPinnedWaitStride = 4;

struct ReqPlan {
  bool all_layers = false, hkvd = false;
  int C = 0, Q = 0, T = 0, N = 0, crit = 0, A = 0, nA = 0;
  std::vector<int32_t> seg_start, seg_delta;
  ChunkOffsets co;
  std::vector<int> Nl;
  RequestLayout rl{};
  HkvdLayout H{};
  float* scores = nullptr;
  int32_t* sel = nullptr;
  __nv_bfloat16* q_crit = nullptr;
  size_t ws_used = 0;
  // The recompute waits for the copy stream every wait_stride layers, each time for the
  // layers up to the next wait: fewer event waits split the programmatic launch chain,
  // at the price of waiting for up to wait_stride - 1 later layers' copies.  1 where the
  // copies are the slow side (files).
  int wait_stride = 1;
};

// Validates a request and carves its buffers from ws.
static qcf_status request_plan(const qcf_model* m, const qcf_request* r, const qcf_outputs* out, void* ws,
                               size_t ws_bytes, ReqPlan* P) {
  qcf_status s = check_model(m, "qcf_request_prefill");
  if (s != QCF_OK) return s;
  if (!r || !out || !ws || !r->chunk_len || !r->chunk_K_host || !r->chunk_V_host || !r->ids)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_request_prefill: NULL pointer");
  if (!out->K_layers || !out->V_layers || !out->last_logits || !out->first_token)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_request_prefill: outputs need K/V layers, logits and first token");
  const qcf_dims& d = m->dims;
  const int L = d.n_layers;
  if (r->n_chunks <= 0 || r->n_chunks > kMaxReqChunks || r->query_len <= 0 || r->crit_layer < 0 ||
      r->crit_layer >= L || r->ratio_bp < 0 || r->ratio_bp > 10000 || r->n_anchor < 0)
    return set_error(QCF_ERR_SHAPE, "qcf_request_prefill: n_chunks=%d query_len=%d crit=%d ratio_bp=%d n_anchor=%d",
                     r->n_chunks, r->query_len, r->crit_layer, r->ratio_bp, r->n_anchor);
  if (r->selector < QCF_SELECT_CRITICAL || r->selector > QCF_SELECT_HKVD)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_request_prefill: unknown selector %d", r->selector);
  const bool all_layers = r->selector == QCF_SELECT_ALL_LAYERS;
  const bool hkvd = r->selector == QCF_SELECT_HKVD;
  std::vector<int32_t> seg_start(r->n_chunks + 1, 0), seg_delta(r->n_chunks, 0);
  ChunkOffsets co;
  co.n_chunks = r->n_chunks;
  for (int c = 0; c < r->n_chunks; ++c) {
    const int len = r->chunk_len[c];
    if (len <= 0 || len < r->n_anchor || !r->chunk_K_host[c] || !r->chunk_V_host[c])
      return set_error(QCF_ERR_SHAPE, "qcf_request_prefill: chunk %d length %d / host pointers", c, len);
    seg_delta[c] = seg_start[c];
    co.off[c] = seg_start[c];
    seg_start[c + 1] = seg_start[c] + len;
  }
  const int C = seg_start[r->n_chunks], Q = r->query_len, T = C + Q;
  int N = 0;
  qcf_num_selected(C, r->ratio_bp, &N);
  // probe depth: the critical layer (QCLast: L-1); QCAll probes L-1 layers and profiles all L;
  // HKVD has no probe (layer 0's keys are then simply copied first)
  const int crit = hkvd ? 0 : (all_layers ? L - 1 : r->crit_layer);
  const int A = r->n_anchor;
  const int nA = (!hkvd && crit > 0) ? A * r->n_chunks : 0;
  std::vector<int> Nl;
  if (hkvd && !hkvd_counts(r->layer_ratio_bp, L, C, r->ratio_bp, &Nl))
    return set_error(QCF_ERR_INVALID_ARG,
                     "qcf_request_prefill: HKVD needs layer_ratio_bp[L] in [0,10000], non-increasing, last == ratio_bp");
  if (nA > 0 && (!r->anchor_K_host || !r->anchor_V_host))
    return set_error(QCF_ERR_INVALID_ARG, "qcf_request_prefill: anchor stores are NULL");
  if (m->rope.max_pos < T) return set_error(QCF_ERR_SHAPE, "qcf_request_prefill: RoPE table %d shorter than T=%d", m->rope.max_pos, T);
  for (int l = 0; l < L; ++l)
    if (!out->K_layers[l] || !out->V_layers[l] || !aligned16(out->K_layers[l]) || !aligned16(out->V_layers[l]))
      return set_error(QCF_ERR_ALIGN, "qcf_request_prefill: fused cache of layer %d NULL or misaligned", l);
  if (take_fault(4) || !aligned16(ws)) return set_error(QCF_ERR_ALIGN, "qcf_request_prefill: workspace misaligned");
  if (take_fault(1)) return set_error(QCF_ERR_INVALID_ARG, "qcf_request_prefill: injected invalid index table");
  Carve cv{static_cast<uint8_t*>(ws), ws_bytes};
  RequestLayout rl{};
  HkvdLayout H{};
  const bool carved = hkvd ? carve_hkvd(cv, d, C, Q, Nl, &H) : carve_request(cv, d, C, Q, nA, N, r->n_chunks, crit, A, &rl);
  if (take_fault(2) || !carved)
    return set_error(QCF_ERR_WORKSPACE, "qcf_request_prefill: workspace %zu too small (need %zu)", ws_bytes, cv.used);
  P->all_layers = all_layers;
  P->hkvd = hkvd;
  P->C = C; P->Q = Q; P->T = T; P->N = N; P->crit = crit; P->A = A; P->nA = nA;
  P->seg_start = std::move(seg_start);
  P->seg_delta = std::move(seg_delta);
  P->co = co;
  P->Nl = std::move(Nl);
  P->rl = rl;
  P->H = H;
  P->scores = out->scores ? out->scores : (hkvd ? H.dev : rl.scores);
  P->sel = out->sel ? out->sel : rl.sel;
  P->q_crit = out->q_crit ? reinterpret_cast<__nv_bfloat16*>(out->q_crit) : rl.q_crit;
  P->ws_used = cv.used;
  return QCF_OK;

}

// Host-to-device copies of the request's anchor stores for the probe layers.
static qcf_status request_copy_anchors(const qcf_model* m, const qcf_request* r, const ReqPlan& P, cudaStream_t xs) {
  const qcf_dims& d = m->dims;
  const int nA = P.nA, crit = P.crit, A = P.A;
  const RequestLayout& rl = P.rl;
  const size_t HD = static_cast<size_t>(d.n_kv_heads) * d.head_dim;
  const size_t eb = sizeof(qcf_bf16);
  cudaError_t e = cudaSuccess;
  for (int c = 0; c < r->n_chunks && nA > 0; ++c) {
    const size_t n_el = static_cast<size_t>(crit) * A * HD;
    if ((e = cudaMemcpyAsync(rl.stK + c * n_el, r->anchor_K_host[c], n_el * eb, cudaMemcpyHostToDevice, xs)) != cudaSuccess ||
        (e = cudaMemcpyAsync(rl.stV + c * n_el, r->anchor_V_host[c], n_el * eb, cudaMemcpyHostToDevice, xs)) != cudaSuccess)
      return cuda_error(e, "qcf_request_prefill: anchor copy");
  }
  return QCF_OK;
}

// The request's chunk K/V of every layer straight into its fused cache, each layer's
// keys re-rotated to their offsets on the copy stream right after they land: with
// crit_part the critical layer's keys (then ev_crit), else every layer in order (the
// critical layer's values only), each followed by ev_layer[l].
static qcf_status request_copy_layers(const qcf_model* m, const qcf_request* r, const qcf_outputs* out,
                                      const ReqPlan& P, cudaStream_t xs, cudaEvent_t ev_crit,
                                      const cudaEvent_t* ev_layer, bool crit_part) {
  const qcf_dims& d = m->dims;
  const int L = d.n_layers, C = P.C, crit = P.crit;
  const std::vector<int32_t>& seg_start = P.seg_start;
  const std::vector<int32_t>& seg_delta = P.seg_delta;
  const size_t HD = static_cast<size_t>(d.n_kv_heads) * d.head_dim;
  const size_t eb = sizeof(qcf_bf16);
  cudaError_t e = cudaSuccess;
  auto copy_layer = [&](int l, bool keys, bool values) -> cudaError_t {
    for (int c = 0; c < r->n_chunks; ++c) {
      const int len = r->chunk_len[c];
      const size_t n_el = static_cast<size_t>(len) * HD;
      const size_t src_off = static_cast<size_t>(l) * n_el;
      const size_t dst_off = static_cast<size_t>(seg_start[c]) * HD;
      cudaError_t ce;
      if (keys && (ce = cudaMemcpyAsync(out->K_layers[l] + dst_off, r->chunk_K_host[c] + src_off, n_el * eb,
                                        cudaMemcpyHostToDevice, xs)) != cudaSuccess)
        return ce;
      if (values && (ce = cudaMemcpyAsync(out->V_layers[l] + dst_off, r->chunk_V_host[c] + src_off, n_el * eb,
                                          cudaMemcpyHostToDevice, xs)) != cudaSuccess)
        return ce;
    }
    return cudaSuccess;
  };
  auto rotate_layer = [&](int l) -> cudaError_t {
    __nv_bfloat16* Kl = reinterpret_cast<__nv_bfloat16*>(out->K_layers[l]);
    return launch_reposition(Kl, Kl, C, d.n_kv_heads, d.head_dim, seg_start.data(), seg_delta.data(), r->n_chunks,
                             &m->rope, xs);
  };
  if (crit_part) {
    if ((e = copy_layer(crit, true, false)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: critical-layer copy");
    if ((e = rotate_layer(crit)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: reposition");
    if ((e = cudaEventRecord(ev_crit, xs)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: record");
    return QCF_OK;
  }
  for (int l = 0; l < L; ++l) {
    if ((e = copy_layer(l, l != crit, true)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: layer copy");
    if (l != crit && (e = rotate_layer(l)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: reposition");
    if ((e = cudaEventRecord(ev_layer[l], xs)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: record");
  }

  return QCF_OK;
}

// ------------------------------------------------------------------ storage tier
//
// Chunk K/V read from files layer by layer (QCFuse 2.A keeps chunk KV on SSD and loads
// layer i+1 while layer i is recomputed).  Reads run as host functions on the copy
// stream, so each one starts once the copy stream reaches it: it fills one half of a
// pinned double buffer, the next operations copy that half to the fused cache, and
// the read two layers later reuses it only after those copies completed (stream
// order).  Meanwhile the compute stream recomputes the layers already landed.
struct StorageCtx {
  std::vector<qcf_chunk_file> files;
  std::vector<int32_t> len;
  size_t row_bytes = 0;
  size_t C = 0;
  uint8_t* buf[2] = {nullptr, nullptr};   // each: C rows of keys, then C rows of values
  int err = 0;                            // first failure (errno, or EIO for a short read)
};
struct StorageRead {
  StorageCtx* ctx;
  int layer, buf;
  bool keys, values, last;
};
static std::atomic<int> g_storage_err{0};

static int read_full(int fd, uint8_t* dst, size_t bytes, int64_t offset) {
  while (bytes > 0) {
    const ssize_t got = pread(fd, dst, bytes, static_cast<off_t>(offset));
    if (got < 0) {
      if (errno == EINTR) continue;
      return errno ? errno : EIO;
    }
    if (got == 0) return EIO;  // the file ends before the block
    dst += got;
    bytes -= static_cast<size_t>(got);
    offset += got;
  }
  return 0;
}

// A pool of reader threads: one layer's blocks (a chunk's keys or values each, in pieces
// of at most kReadPiece bytes) are read concurrently, so a storage device sees several
// requests in flight and page-cache copies use several cores.
class ReadPool {
 public:
  static ReadPool& get() {
    static ReadPool pool;
    return pool;
  }
  // Runs every task on the pool and returns when all are done.
  void run(std::vector<std::function<void()>>& tasks) {
    std::unique_lock<std::mutex> lk(mu_);
    for (auto& t : tasks) queue_.push_back(&t);
    pending_ += tasks.size();
    cv_.notify_all();
    done_cv_.wait(lk, [&] { return pending_ == 0; });
  }

 private:
  ReadPool() {
    const unsigned hw = std::thread::hardware_concurrency();
    const int n = hw >= 16 ? 16 : (hw >= 8 ? static_cast<int>(hw) : 8);
    for (int i = 0; i < n; ++i) threads_.emplace_back([this] { work(); });
  }
  ~ReadPool() {
    {
      std::lock_guard<std::mutex> lk(mu_);
      stop_ = true;
    }
    cv_.notify_all();
    for (auto& t : threads_) t.join();
  }
  void work() {
    std::unique_lock<std::mutex> lk(mu_);
    while (true) {
      cv_.wait(lk, [&] { return stop_ || !queue_.empty(); });
      if (stop_ && queue_.empty()) return;
      std::function<void()>* t = queue_.back();
      queue_.pop_back();
      lk.unlock();
      (*t)();
      lk.lock();
      if (--pending_ == 0) done_cv_.notify_all();
    }
  }
  std::mutex mu_;
  std::condition_variable cv_, done_cv_;
  std::vector<std::function<void()>*> queue_;
  size_t pending_ = 0;
  bool stop_ = false;
  std::vector<std::thread> threads_;
};

// Read pieces: page-cache reads are memory copies, split finely over the threads; direct
// reads go to the device in larger requests (both multiples of the 4096-byte O_DIRECT
// alignment).
constexpr size_t kReadPiece = 256 << 10;
constexpr size_t kReadPieceDirect = 1 << 20;
static size_t read_piece(int fd) {
  const int fl = fcntl(fd, F_GETFL);
  return fl != -1 && (fl & O_DIRECT) ? kReadPieceDirect : kReadPiece;
}

static void CUDART_CB storage_read_fn(void* arg) {
  StorageRead* rd = static_cast<StorageRead*>(arg);
  StorageCtx* c = rd->ctx;
  if (c->err == 0 && (rd->keys || rd->values)) {
    std::vector<std::function<void()>> tasks;
    size_t n_pieces = 0;
    for (size_t i = 0; i < c->files.size(); ++i)
      n_pieces += 2 * ((static_cast<size_t>(c->len[i]) * c->row_bytes + kReadPiece - 1) / kReadPiece);
    std::vector<int> errs(n_pieces, 0);
    size_t row0 = 0, piece = 0;
    auto add = [&](int fd, uint8_t* dst, size_t bytes, int64_t off) {
      const size_t step = read_piece(fd);
      for (size_t done = 0; done < bytes; done += step) {
        const size_t n = bytes - done < step ? bytes - done : step;
        int* err = &errs[piece++];
        tasks.emplace_back([=] { *err = read_full(fd, dst + done, n, off + static_cast<int64_t>(done)); });
      }
    };
    for (size_t i = 0; i < c->files.size(); ++i) {
      const qcf_chunk_file f = c->files[i];
      const size_t bytes = static_cast<size_t>(c->len[i]) * c->row_bytes;
      const int64_t layer_off = static_cast<int64_t>(rd->layer) * f.layer_stride;
      if (rd->keys) add(f.fd, c->buf[rd->buf] + row0 * c->row_bytes, bytes, f.k_offset + layer_off);
      if (rd->values) add(f.fd, c->buf[rd->buf] + (c->C + row0) * c->row_bytes, bytes, f.v_offset + layer_off);
      row0 += static_cast<size_t>(c->len[i]);
    }
    ReadPool::get().run(tasks);
    for (int e : errs)
      if (e && c->err == 0) c->err = e;
  }
  if (rd->last) {
    if (c->err) {
      int expected = 0;
      g_storage_err.compare_exchange_strong(expected, c->err);
    }
    delete c;
  }
  delete rd;
}

// request_copy_layers with the chunk K/V coming from files through the pinned double buffer.
static qcf_status request_copy_layers_storage(const qcf_model* m, const qcf_outputs* out, const ReqPlan& P,
                                              StorageCtx* ctx, cudaStream_t xs, cudaEvent_t ev_crit,
                                              const cudaEvent_t* ev_layer) {
  const qcf_dims& d = m->dims;
  const int L = d.n_layers, C = P.C, crit = P.crit;
  const size_t HD = static_cast<size_t>(d.n_kv_heads) * d.head_dim;
  const size_t bytes = static_cast<size_t>(C) * HD * sizeof(qcf_bf16);
  int b = 0;
  bool enqueued = false;  // host functions holding ctx are in the stream
  auto enqueue_read = [&](int layer, bool keys, bool values, bool last) -> cudaError_t {
    StorageRead* rd = new StorageRead{ctx, layer, b, keys, values, last};
    const cudaError_t e = cudaLaunchHostFunc(xs, storage_read_fn, rd);
    if (e != cudaSuccess) delete rd;
    else enqueued = true;
    return e;
  };
  // On a failed enqueue: with no host function holding ctx it is freed here; otherwise the
  // final host function frees it after the ones before (if even that cannot be enqueued,
  // ctx is left allocated rather than freed under a pending host function).
  auto fail = [&](cudaError_t e, const char* what) {
    if (!enqueued) delete ctx;
    else enqueue_read(0, false, false, true);
    return cuda_error(e, what);
  };
  auto rotate = [&](int l) -> cudaError_t {
    __nv_bfloat16* Kl = reinterpret_cast<__nv_bfloat16*>(out->K_layers[l]);
    return launch_reposition(Kl, Kl, C, d.n_kv_heads, d.head_dim, P.seg_start.data(), P.seg_delta.data(),
                             static_cast<int>(P.seg_start.size()) - 1, &m->rope, xs);
  };
  cudaError_t e;
  if ((e = enqueue_read(crit, true, false, false)) != cudaSuccess) return fail(e, "storage: read");
  if ((e = cudaMemcpyAsync(out->K_layers[crit], ctx->buf[b], bytes, cudaMemcpyHostToDevice, xs)) != cudaSuccess)
    return fail(e, "storage: copy");
  if ((e = rotate(crit)) != cudaSuccess) return fail(e, "storage: reposition");
  if ((e = cudaEventRecord(ev_crit, xs)) != cudaSuccess) return fail(e, "storage: record");
  for (int l = 0; l < L; ++l) {
    b ^= 1;
    const bool keys = l != crit;
    if ((e = enqueue_read(l, keys, true, false)) != cudaSuccess) return fail(e, "storage: read");
    if (keys && (e = cudaMemcpyAsync(out->K_layers[l], ctx->buf[b], bytes, cudaMemcpyHostToDevice, xs)) != cudaSuccess)
      return fail(e, "storage: copy");
    if ((e = cudaMemcpyAsync(out->V_layers[l], ctx->buf[b] + bytes, bytes, cudaMemcpyHostToDevice, xs)) != cudaSuccess)
      return fail(e, "storage: copy");
    if (keys && (e = rotate(l)) != cudaSuccess) return fail(e, "storage: reposition");
    if ((e = cudaEventRecord(ev_layer[l], xs)) != cudaSuccess) return fail(e, "storage: record");
  }
  // the last host function reports a failed read and frees the context
  if ((e = enqueue_read(0, false, false, true)) != cudaSuccess) return fail(e, "storage: read");
  return QCF_OK;
}

// The compute stream of one request: probe, profile and selection (or the
// KV-deviation filter), the per-layer recompute waiting on ev_layer[l], LM head.
// enqueue_layers (may be empty) puts the per-layer copies, and their ev_layer records, on
// the copy stream; it runs once, before the first wait on any ev_layer[l] is enqueued, and
// as late as that allows: after the probe, whose launches then reach the GPU without
// waiting behind the host's many copy calls.
static qcf_status request_compute(const qcf_model* m, const qcf_request* r, const qcf_outputs* out, ReqPlan& P,
                                  cudaStream_t cs, cudaEvent_t ev_anchor, cudaEvent_t ev_crit,
                                  const cudaEvent_t* ev_layer,
                                  const std::function<qcf_status()>& enqueue_layers = {},
                                  bool probe_done = false) {
  const qcf_dims& d = m->dims;
  const int L = d.n_layers;
  const bool all_layers = P.all_layers, hkvd = P.hkvd;
  const int C = P.C, Q = P.Q, T = P.T, N = P.N, crit = P.crit, A = P.A, nA = P.nA;
  const std::vector<int>& Nl = P.Nl;
  const ChunkOffsets& co = P.co;
  RequestLayout& rl = P.rl;
  HkvdLayout& H = P.H;
  float* scores = P.scores;
  int32_t* sel = P.sel;
  __nv_bfloat16* q_crit = P.q_crit;
  qcf_status s = QCF_OK;
  cudaError_t e = cudaSuccess;
  // ---- compute stream
  LayerBufs& glb = hkvd ? H.lb : rl.lb;
  if ((s = gemm_ws_prepare(glb.gemm_ws, glb.gemm_ws_bytes, cs)) != QCF_OK) return s;
  glb.gemm_zeroed = true;
  const __nv_bfloat16* embed = reinterpret_cast<const __nv_bfloat16*>(m->embed);
  const float* x_final = nullptr;  // final hidden states of the recomputed rows [ns][d]
  int ns = 0;
  bool layers_enqueued = !enqueue_layers;
  auto layers_now = [&]() -> qcf_status {
    if (layers_enqueued) return QCF_OK;
    layers_enqueued = true;
    return enqueue_layers();
  };
  if (hkvd) {
    if ((s = layers_now()) != QCF_OK) return s;
    // every context row and the query enter layer 0; the kept set shrinks layer by layer
    {
      LaunchScope ls(KC_MISC, cs);
      iota_kernel<<<(T + 255) / 256, 256, 0, cs>>>(H.rows_a, T, 0);
      iota_kernel<<<(T + 255) / 256, 256, 0, cs>>>(H.iota, T, 0);
    }
    if ((e = launch_embed(embed, d.vocab, d.d_model, r->ids, nullptr, 0, T, H.x_a, cs)) != cudaSuccess)
      return cuda_error(e, "qcf_request_prefill: embed");
    float* xp = H.x_a;
    float* xn = H.x_b;
    int32_t* rp = H.rows_a;
    int32_t* rn = H.rows_b;
    int n_ctx = C;
    for (int l = 0; l < L; ++l) {
      if ((e = cudaStreamWaitEvent(cs, ev_layer[l], 0)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: wait");
      s = hkvd_layer(m, l, H, xp, rp, n_ctx, Nl[l], xn, rn, reinterpret_cast<__nv_bfloat16*>(out->K_layers[l]),
                     reinterpret_cast<__nv_bfloat16*>(out->V_layers[l]), l == 0 ? scores : nullptr,
                     out->layer_sel ? out->layer_sel + static_cast<size_t>(l) * (H.N0 > 0 ? H.N0 : 1) : nullptr, cs);
      if (s != QCF_OK) return s;
      std::swap(xp, xn);
      std::swap(rp, rn);
      n_ctx = Nl[l];
    }
    if (N > 0 && out->sel &&
        (e = cudaMemcpyAsync(out->sel, rp, N * sizeof(int32_t), cudaMemcpyDeviceToDevice, cs)) != cudaSuccess)
      return cuda_error(e, "qcf_request_prefill: selection copy");
    ns = N + Q;
    x_final = xp;
    if ((e = launch_lm_head(m, xp + static_cast<size_t>(ns - 1) * d.d_model, out->last_logits, out->first_token,
                            H.lm_ws, cs)) != cudaSuccess)
      return cuda_error(e, "qcf_request_prefill: lm head");
  } else {
    const float scale = 1.0f / sqrtf(static_cast<float>(d.head_dim));
    if (all_layers && (e = cudaMemsetAsync(rl.scores_acc, 0, static_cast<size_t>(C) * sizeof(float), cs)) != cudaSuccess)
      return cuda_error(e, "qcf_request_prefill: clear scores");
    if (all_layers && (s = layers_now()) != QCF_OK) return s;   // the probe profiles every layer
    // probe (unless a batch ran it for several requests at once): query rows at positions
    // C..T-1 with the anchors as KV prefix (probe cache rows 0..nA-1), then q at the critical layer
    if (!probe_done) {
      if ((e = launch_embed(embed, d.vocab, d.d_model, r->ids, nullptr, C, Q, rl.x, cs)) != cudaSuccess)
        return cuda_error(e, "qcf_request_prefill: embed");
      {
        LaunchScope ls(KC_MISC, cs);
        iota_kernel<<<(Q + 255) / 256, 256, 0, cs>>>(rl.probe_pos, Q, C);
      }
      {
        LaunchScope ls(KC_MISC, cs);
        iota_kernel<<<(Q + 255) / 256, 256, 0, cs>>>(rl.probe_row, Q, nA);
      }
      if (crit > 0) {
        if ((e = cudaStreamWaitEvent(cs, ev_anchor, 0)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: wait");
        const size_t pstride = static_cast<size_t>(nA + Q) * d.n_kv_heads * d.head_dim;
        if (nA > 0) {
          const long long threads = static_cast<long long>(crit) * nA * d.n_kv_heads * (d.head_dim / 16);
          LaunchScope ls(KC_ROPE, cs);
          anchor_assemble_kernel<<<static_cast<unsigned int>((threads + 255) / 256), 256, 0, cs>>>(
              rl.stK, rl.stV, crit, A, d.n_kv_heads, d.head_dim, m->rope.cos, m->rope.sin, co, rl.pK, rl.pV, pstride);
        }
        for (int l = 0; l < crit; ++l) {
          // consecutive probe layers follow each other directly (QCAll puts a profile and an
          // event wait between them): their first launch is programmatic too
          s = layer_forward_impl(m, l, rl.x, rl.probe_pos, rl.probe_row, Q, rl.pK + l * pstride, rl.pV + l * pstride,
                                 nA + Q, rl.lb, cs, true, !all_layers);
          if (s != QCF_OK) return s;
          if (all_layers) {   // QCAll: this probe layer's q against this layer's re-rotated keys
            if ((e = cudaStreamWaitEvent(cs, ev_layer[l], 0)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: wait");
            s = qcf_profile_scores(reinterpret_cast<const qcf_bf16*>(rl.lb.q), out->K_layers[l], Q, C, d.n_heads,
                                   d.n_kv_heads, d.head_dim, scale, rl.scores_tmp, rl.prof_ws, rl.prof_ws_bytes, cs);
            if (s != QCF_OK) return s;
            LaunchScope ls(KC_MISC, cs);
            add_f32_kernel<<<(C + 255) / 256, 256, 0, cs>>>(rl.scores_acc, rl.scores_tmp, C);
          }
        }
      }
      // critical layer: q = RoPE(RMSNorm(x) W_q) only
      {
        const qcf_layer_weights& w = m->layers[crit];
        // programmatic when it follows the last probe layer's down projection directly
        if ((e = launch_rmsnorm(rl.x, Q, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.g_attn), d.eps, rl.lb.h, cs,
                                crit > 0 && !all_layers && Q <= kPdlMaxRows)) != cudaSuccess)
          return cuda_error(e, "qcf_request_prefill: rmsnorm");
        EpiParams ep{};
        ep.q_out = q_crit;
        ep.rope_pos = rl.probe_pos;
        ep.cache_row = nullptr;
        ep.cos_t = m->rope.cos;
        ep.sin_t = m->rope.sin;
        ep.Hq = d.n_heads;
        ep.Hkv = d.n_kv_heads;
        ep.D = d.head_dim;
        ep.T = 1;
        ep.max_pos = m->rope.max_pos;
        ep.status = device_status_ptr();
        s = gemm_launch(EPI_QKV_ROPE, rl.lb.h, Q, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.w_qkv),
                        d.n_heads * d.head_dim, ep, rl.lb.gemm_ws, rl.lb.gemm_ws_bytes, cs, KC_GEMM_PROBE, false, Q <= kPdlMaxRows,
                        rl.lb.gemm_zeroed);
        if (s != QCF_OK) return s;
      }
    }  // probe
    if ((s = layers_now()) != QCF_OK) return s;
    // profile the re-rotated critical-layer keys and select
    if ((e = cudaStreamWaitEvent(cs, ev_crit, 0)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: wait");
    __nv_bfloat16* Kcrit = reinterpret_cast<__nv_bfloat16*>(out->K_layers[crit]);
    s = qcf_profile_scores(reinterpret_cast<const qcf_bf16*>(q_crit), reinterpret_cast<const qcf_bf16*>(Kcrit), Q, C,
                           d.n_heads, d.n_kv_heads, d.head_dim, scale, scores, rl.prof_ws, rl.prof_ws_bytes, cs);
    if (s != QCF_OK) return s;
    if (all_layers) {
      LaunchScope ls(KC_MISC, cs);
      add_f32_kernel<<<(C + 255) / 256, 256, 0, cs>>>(scores, rl.scores_acc, C);
    }
    if (N > 0) {
      if (r->forced_sel) {
        if ((e = cudaMemcpyAsync(sel, r->forced_sel, N * sizeof(int32_t), cudaMemcpyDeviceToDevice, cs)) != cudaSuccess)
          return cuda_error(e, "qcf_request_prefill: forced selection");
      } else {
        // above 16384 context tokens the selection spreads over a cooperative grid
        s = rl.topn_ws_bytes > 0 ? qcf_topn_select_ws(scores, C, N, sel, rl.topn_ws, rl.topn_ws_bytes, cs)
                                 : topn_launch(scores, C, N, sel, cs, true);
        if (s != QCF_OK) return s;
      }
    }
    ns = N + Q;
    {
      LaunchScope ls(KC_MISC, cs);
      if ((e = launch_pdl(make_rows_kernel, dim3((ns + 255) / 256), dim3(256), 0, cs, static_cast<const int32_t*>(sel), N,
                          C, ns, rl.rows)) != cudaSuccess)
        return cuda_error(e, "qcf_request_prefill: rows");
    }
    // pipelined per-layer recompute of the selected rows and the query
    if ((e = launch_embed(embed, d.vocab, d.d_model, r->ids, rl.rows, 0, ns, rl.x, cs, true)) != cudaSuccess)
      return cuda_error(e, "qcf_request_prefill: embed");
    const int stride = std::max(1, P.wait_stride);
    for (int l = 0; l < L; ++l) {
      const bool wait_here = l % stride == 0;
      if (wait_here && (e = cudaStreamWaitEvent(cs, ev_layer[std::min(l + stride - 1, L - 1)], 0)) != cudaSuccess)
        return cuda_error(e, "qcf_request_prefill: wait");
      __nv_bfloat16* Kl = reinterpret_cast<__nv_bfloat16*>(out->K_layers[l]);
      __nv_bfloat16* Vl = reinterpret_cast<__nv_bfloat16*>(out->V_layers[l]);
      s = layer_forward_impl(m, l, rl.x, rl.rows, rl.rows, ns, Kl, Vl, T, rl.lb, cs, false, !wait_here);
      if (s != QCF_OK) return s;
    }
    if ((e = launch_lm_head(m, rl.x + static_cast<size_t>(ns - 1) * d.d_model, out->last_logits, out->first_token,
                            rl.lm_ws, cs, ns <= kPdlMaxRows)) != cudaSuccess)
      return cuda_error(e, "qcf_request_prefill: lm head");
    x_final = rl.x;
  }
  if (out->x_rows &&
      (e = cudaMemcpyAsync(out->x_rows, x_final, static_cast<size_t>(ns) * d.d_model * sizeof(float),
                           cudaMemcpyDeviceToDevice, cs)) != cudaSuccess)
    return cuda_error(e, "qcf_request_prefill: copy rows");
  if (out->first_token_host &&
      (e = cudaMemcpyAsync(out->first_token_host, out->first_token, sizeof(int32_t), cudaMemcpyDeviceToHost, cs)) !=
          cudaSuccess)
    return cuda_error(e, "qcf_request_prefill: first token copy");
  return QCF_OK;
}

// ------------------------------------------------------------------ batches with shared chunks

constexpr int kMaxBatch = 64;

// The distinct chunks of a batch (the same host K and V arrays and length; a content-keyed
// chunk store hands equal chunks the same arrays) and where each request's chunk slots
// point in the shared staging rows.
struct UniqueChunks {
  std::vector<const qcf_bf16*> K, V;
  std::vector<int> len, start;            // staging rows [start, start + len)
  int rows = 0;
  std::vector<std::vector<int>> of_req;   // [request][chunk slot] -> distinct chunk
};

static bool unique_chunks(const qcf_request* reqs, int n_req, UniqueChunks* U) {
  std::map<std::tuple<const void*, const void*, int>, int> idx;
  U->of_req.assign(n_req, {});
  for (int i = 0; i < n_req; ++i) {
    const qcf_request& r = reqs[i];
    if (r.n_chunks <= 0 || !r.chunk_len || !r.chunk_K_host || !r.chunk_V_host) return false;
    for (int c = 0; c < r.n_chunks; ++c) {
      const auto key = std::make_tuple(static_cast<const void*>(r.chunk_K_host[c]),
                                       static_cast<const void*>(r.chunk_V_host[c]), r.chunk_len[c]);
      auto it = idx.find(key);
      int u;
      if (it == idx.end()) {
        u = static_cast<int>(U->K.size());
        idx.emplace(key, u);
        U->K.push_back(r.chunk_K_host[c]);
        U->V.push_back(r.chunk_V_host[c]);
        U->len.push_back(r.chunk_len[c]);
        U->start.push_back(U->rows);
        U->rows += r.chunk_len[c];
      } else {
        u = it->second;
      }
      U->of_req[i].push_back(u);
    }
  }
  return true;
}

struct BatchStaging {
  __nv_bfloat16* K[2];   // [rows][HD] per layer parity
  __nv_bfloat16* V[2];
  __nv_bfloat16* Kc;     // critical-layer keys
  std::vector<int32_t*> src_row, delta;   // per request [C]
};

static bool carve_staging(Carve& c, const qcf_dims& d, const UniqueChunks& U, const std::vector<int>& Cs,
                          BatchStaging* B) {
  const size_t n = static_cast<size_t>(U.rows) * d.n_kv_heads * d.head_dim;
  for (int b = 0; b < 2; ++b) {
    B->K[b] = c.take<__nv_bfloat16>(n);
    B->V[b] = c.take<__nv_bfloat16>(n);
  }
  B->Kc = c.take<__nv_bfloat16>(n);
  B->src_row.clear();
  B->delta.clear();
  for (int C : Cs) {
    B->src_row.push_back(c.take<int32_t>(C));
    B->delta.push_back(c.take<int32_t>(C));
  }
  return c.ok;
}

}  // namespace qcf

using namespace qcf;

// ------------------------------------------------------------------ merged probe of a batch
//
// Requests of a batch that share their critical layer (QCFuse selector, head dim 128) run
// the probe together: their query rows, each request's padded to whole attention row
// blocks, go through the probe layers as one row set, so each probe layer's weights
// stream once for the group instead of once per request.  Each request keeps its anchors
// and query K/V in its own segment of one probe cache, and each attention row block reads
// keys from its own request's segment only.  A group holds at most 128 rows: the GEMMs
// then take the plan of a single request's probe and every row is computed as in its own
// request's probe, so each request's q at the critical layer is bitwise what it would be
// alone.
constexpr int kMergedProbeRows = 128;

struct MergedProbeMeta {
  int n;
  int C[kMaxBatch], Q[kMaxBatch], nA[kMaxBatch], roff[kMaxBatch], seg[kMaxBatch];
};

// Row tables of a merged probe: RoPE position (a padding row repeats its request's last
// query position), cache row in the shared probe cache, and each row block's key base.
__global__ void merged_probe_tables_kernel(const MergedProbeMeta meta, int M, int BR, int32_t* __restrict__ pos,
                                           int32_t* __restrict__ row, int32_t* __restrict__ key0) {
  const int mr = blockIdx.x * blockDim.x + threadIdx.x;
  if (mr >= M) return;
  int i = 0;
  while (i + 1 < meta.n && meta.roff[i + 1] <= mr) ++i;
  const int j = mr - meta.roff[i];
  pos[mr] = meta.C[i] + min(j, meta.Q[i] - 1);
  row[mr] = meta.seg[i] + meta.nA[i] + j;
  if (mr % BR == 0) key0[mr / BR] = meta.seg[i];
}

struct MergedProbe {
  std::vector<int> members;   // request indices
  MergedProbeMeta meta{};
  int M = 0, S = 0, crit = 0;
  float* x = nullptr;
  int32_t *pos = nullptr, *row = nullptr, *key0 = nullptr;
  __nv_bfloat16 *pK = nullptr, *pV = nullptr, *q = nullptr;
  LayerBufs lb{};
};

// Groups of requests whose probes merge (consecutive requests with the same critical layer,
// at most kMergedProbeRows padded rows per group); requests in no group of two or more
// run their own probe.
static std::vector<MergedProbe> merged_probe_groups(const qcf_dims& d, const qcf_request* reqs, int n_req) {
  std::vector<MergedProbe> groups;
  if (d.head_dim != 128 || d.n_heads % d.n_kv_heads) return groups;
  const int BR = 128 / (d.n_heads / d.n_kv_heads);
  MergedProbe cur;
  auto flush = [&]() {
    if (cur.members.size() >= 2) groups.push_back(cur);
    cur = MergedProbe{};
  };
  for (int i = 0; i < n_req; ++i) {
    const qcf_request& r = reqs[i];
    const bool ok = r.selector == QCF_SELECT_CRITICAL && r.crit_layer > 0 && r.query_len > 0;
    const int Qp = ok ? (r.query_len + BR - 1) / BR * BR : 0;
    if (!ok || Qp > kMergedProbeRows) {
      flush();
      continue;
    }
    if (!cur.members.empty() && (cur.crit != r.crit_layer || cur.M + Qp > kMergedProbeRows)) flush();
    const int k = static_cast<int>(cur.members.size());
    int C = 0;
    for (int c = 0; c < r.n_chunks; ++c) C += r.chunk_len[c];
    const int nA = r.n_anchor * r.n_chunks;
    cur.crit = r.crit_layer;
    cur.meta.C[k] = C;
    cur.meta.Q[k] = r.query_len;
    cur.meta.nA[k] = nA;
    cur.meta.roff[k] = cur.M;
    cur.meta.seg[k] = cur.S;
    cur.meta.n = k + 1;
    cur.M += Qp;
    cur.S += nA + Qp;
    cur.members.push_back(i);
  }
  flush();
  return groups;
}

static bool carve_merged_probe(Carve& c, const qcf_dims& d, MergedProbe* g) {
  const int BR = 128 / (d.n_heads / d.n_kv_heads);
  const size_t HD = static_cast<size_t>(d.n_kv_heads) * d.head_dim;
  g->x = c.take<float>(static_cast<size_t>(g->M) * d.d_model);
  g->pos = c.take<int32_t>(g->M);
  g->row = c.take<int32_t>(g->M);
  g->key0 = c.take<int32_t>(g->M / BR);
  g->pK = c.take<__nv_bfloat16>(static_cast<size_t>(g->crit) * g->S * HD);
  g->pV = c.take<__nv_bfloat16>(static_cast<size_t>(g->crit) * g->S * HD);
  g->q = c.take<__nv_bfloat16>(static_cast<size_t>(g->M) * d.n_heads * d.head_dim);
  return carve_layer(c, d, g->M, g->S, &g->lb);
}

// The probe of one merged group, up to each member's q at the critical layer (written to
// the member's own q_crit buffer).
static qcf_status run_merged_probe(const qcf_model* m, const qcf_request* reqs, const std::vector<ReqPlan>& P,
                                   MergedProbe& g, cudaStream_t cs, cudaEvent_t ev_anchor) {
  const qcf_dims& d = m->dims;
  const int BR = 128 / (d.n_heads / d.n_kv_heads), crit = g.crit;
  const size_t HD = static_cast<size_t>(d.n_kv_heads) * d.head_dim;
  const size_t pstride = static_cast<size_t>(g.S) * HD;
  const size_t qrow = static_cast<size_t>(d.n_heads) * d.head_dim;
  const __nv_bfloat16* embed = reinterpret_cast<const __nv_bfloat16*>(m->embed);
  qcf_status s = gemm_ws_prepare(g.lb.gemm_ws, g.lb.gemm_ws_bytes, cs);
  if (s != QCF_OK) return s;
  g.lb.gemm_zeroed = true;
  cudaError_t e;
  {
    LaunchScope ls(KC_MISC, cs);
    merged_probe_tables_kernel<<<(g.M + 127) / 128, 128, 0, cs>>>(g.meta, g.M, BR, g.pos, g.row, g.key0);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_error(e, "qcf_batch_prefill: probe tables");
  }
  for (int k = 0; k < g.meta.n; ++k) {   // each member's query tokens (padding rows repeat the last)
    const int Qp = (g.meta.Q[k] + BR - 1) / BR * BR;
    if ((e = launch_embed(embed, d.vocab, d.d_model, reqs[g.members[k]].ids, g.pos + g.meta.roff[k], 0, Qp,
                          g.x + static_cast<size_t>(g.meta.roff[k]) * d.d_model, cs)) != cudaSuccess)
      return cuda_error(e, "qcf_batch_prefill: embed");
  }
  if ((e = cudaStreamWaitEvent(cs, ev_anchor, 0)) != cudaSuccess) return cuda_error(e, "qcf_batch_prefill: wait");
  for (int k = 0; k < g.meta.n; ++k) {   // each member's anchor rows at the start of its segment
    const ReqPlan& p = P[g.members[k]];
    if (p.nA == 0) continue;
    const long long threads = static_cast<long long>(crit) * p.nA * d.n_kv_heads * (d.head_dim / 16);
    LaunchScope ls(KC_ROPE, cs);
    anchor_assemble_kernel<<<static_cast<unsigned int>((threads + 255) / 256), 256, 0, cs>>>(
        p.rl.stK, p.rl.stV, crit, p.A, d.n_kv_heads, d.head_dim, m->rope.cos, m->rope.sin, p.co,
        g.pK + static_cast<size_t>(g.meta.seg[k]) * HD, g.pV + static_cast<size_t>(g.meta.seg[k]) * HD, pstride);
  }
  for (int l = 0; l < crit; ++l) {
    s = layer_forward_impl(m, l, g.x, g.pos, g.row, g.M, g.pK + l * pstride, g.pV + l * pstride, g.S, g.lb, cs, true,
                           l > 0, g.key0);
    if (s != QCF_OK) return s;
  }
  const qcf_layer_weights& w = m->layers[crit];
  if ((e = launch_rmsnorm(g.x, g.M, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.g_attn), d.eps, g.lb.h, cs,
                          true)) != cudaSuccess)
    return cuda_error(e, "qcf_batch_prefill: rmsnorm");
  EpiParams ep{};
  ep.q_out = g.q;
  ep.rope_pos = g.pos;
  ep.cache_row = nullptr;
  ep.cos_t = m->rope.cos;
  ep.sin_t = m->rope.sin;
  ep.Hq = d.n_heads;
  ep.Hkv = d.n_kv_heads;
  ep.D = d.head_dim;
  ep.T = 1;
  ep.max_pos = m->rope.max_pos;
  ep.status = device_status_ptr();
  s = gemm_launch(EPI_QKV_ROPE, g.lb.h, g.M, d.d_model, reinterpret_cast<const __nv_bfloat16*>(w.w_qkv),
                  d.n_heads * d.head_dim, ep, g.lb.gemm_ws, g.lb.gemm_ws_bytes, cs, KC_GEMM_PROBE, false, true,
                  g.lb.gemm_zeroed);
  if (s != QCF_OK) return s;
  for (int k = 0; k < g.meta.n; ++k) {
    const ReqPlan& p = P[g.members[k]];
    if ((e = cudaMemcpyAsync(p.q_crit, g.q + static_cast<size_t>(g.meta.roff[k]) * qrow,
                             static_cast<size_t>(p.Q) * qrow * sizeof(__nv_bfloat16), cudaMemcpyDeviceToDevice, cs)) !=
        cudaSuccess)
      return cuda_error(e, "qcf_batch_prefill: q copy");
  }
  return QCF_OK;
}

extern "C" {

size_t qcf_layer_workspace_size(const qcf_dims* dims, int n, int T) {
  if (!dims || n <= 0 || T <= 0) return 0;
  return layer_ws_bytes(*dims, n, T);
}

qcf_status qcf_fused_layer_forward(const qcf_model* m, int layer, float* x, const int32_t* rope_pos,
                                   const int32_t* cache_row, int n, qcf_bf16* K_cache, qcf_bf16* V_cache, int T,
                                   void* ws, size_t ws_bytes, void* stream) {
  qcf_status s = check_model(m, "qcf_fused_layer_forward");
  if (s != QCF_OK) return s;
  if (!x || !rope_pos || !cache_row || !K_cache || !V_cache || !ws)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_fused_layer_forward: NULL pointer");
  if (layer < 0 || layer >= m->dims.n_layers || n < 0 || T <= 0 || n > T)
    return set_error(QCF_ERR_SHAPE, "qcf_fused_layer_forward: layer=%d n=%d T=%d", layer, n, T);
  if (m->rope.max_pos < T) return set_error(QCF_ERR_SHAPE, "qcf_fused_layer_forward: RoPE table shorter than T");
  if (take_fault(4) || !aligned16(x) || !aligned16(K_cache) || !aligned16(V_cache) || !aligned16(ws))
    return set_error(QCF_ERR_ALIGN, "qcf_fused_layer_forward: alignment");
  if (take_fault(2) || ws_bytes < layer_ws_bytes(m->dims, n, T))
    return set_error(QCF_ERR_WORKSPACE, "qcf_fused_layer_forward: workspace %zu < %zu", ws_bytes,
                     layer_ws_bytes(m->dims, n, T));
  if (n == 0) return QCF_OK;
  Carve c{static_cast<uint8_t*>(ws), ws_bytes};
  LayerBufs b;
  if (!carve_layer(c, m->dims, n, T, &b)) return set_error(QCF_ERR_WORKSPACE, "qcf_fused_layer_forward: workspace");
  if ((s = gemm_ws_prepare(b.gemm_ws, b.gemm_ws_bytes, static_cast<cudaStream_t>(stream))) != QCF_OK) return s;
  b.gemm_zeroed = true;
  return layer_forward_impl(m, layer, x, rope_pos, cache_row, n, reinterpret_cast<__nv_bfloat16*>(K_cache),
                            reinterpret_cast<__nv_bfloat16*>(V_cache), T, b, static_cast<cudaStream_t>(stream));
}

size_t qcf_full_prefill_workspace_size(const qcf_dims* dims, int T) {
  if (!dims || T <= 0) return 0;
  Carve c{nullptr, 0};
  c.take<float>(static_cast<size_t>(T) * dims->d_model);
  c.take<int32_t>(T);
  c.take<uint8_t>(qcf_lm_head_workspace_size(dims));
  c.take<uint8_t>(layer_ws_bytes(*dims, T, T));
  return c.used;
}

qcf_status qcf_full_prefill(const qcf_model* m, const int32_t* ids, int T, qcf_bf16* const* K_layers,
                            qcf_bf16* const* V_layers, float* last_logits, int32_t* first_token, void* ws,
                            size_t ws_bytes, void* stream) {
  qcf_status s = check_model(m, "qcf_full_prefill");
  if (s != QCF_OK) return s;
  if (!ids || !K_layers || !V_layers || !last_logits || !first_token || !ws)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_full_prefill: NULL pointer");
  if (T <= 0 || m->rope.max_pos < T) return set_error(QCF_ERR_SHAPE, "qcf_full_prefill: T=%d (RoPE table %d)", T, m->rope.max_pos);
  for (int l = 0; l < m->dims.n_layers; ++l)
    if (!K_layers[l] || !V_layers[l] || !aligned16(K_layers[l]) || !aligned16(V_layers[l]))
      return set_error(QCF_ERR_ALIGN, "qcf_full_prefill: layer %d cache pointer NULL or misaligned", l);
  if (take_fault(2) || ws_bytes < qcf_full_prefill_workspace_size(&m->dims, T))
    return set_error(QCF_ERR_WORKSPACE, "qcf_full_prefill: workspace too small");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Carve c{static_cast<uint8_t*>(ws), ws_bytes};
  float* x = c.take<float>(static_cast<size_t>(T) * m->dims.d_model);
  int32_t* pos = c.take<int32_t>(T);
  void* lm_ws = c.take<uint8_t>(qcf_lm_head_workspace_size(&m->dims));
  LayerBufs b;
  if (!carve_layer(c, m->dims, T, T, &b)) return set_error(QCF_ERR_WORKSPACE, "qcf_full_prefill: workspace");
  if ((s = gemm_ws_prepare(b.gemm_ws, b.gemm_ws_bytes, st)) != QCF_OK) return s;
  b.gemm_zeroed = true;
  cudaError_t e = launch_embed(reinterpret_cast<const __nv_bfloat16*>(m->embed), m->dims.vocab, m->dims.d_model, ids,
                               nullptr, 0, T, x, st);
  if (e != cudaSuccess) return cuda_error(e, "qcf_full_prefill: embed");
  {
    LaunchScope ls(KC_MISC, st);
    iota_kernel<<<(T + 255) / 256, 256, 0, st>>>(pos, T, 0);
  }
  for (int l = 0; l < m->dims.n_layers; ++l) {
    s = layer_forward_impl(m, l, x, pos, pos, T, reinterpret_cast<__nv_bfloat16*>(K_layers[l]),
                           reinterpret_cast<__nv_bfloat16*>(V_layers[l]), T, b, st);
    if (s != QCF_OK) return s;
  }
  e = launch_lm_head(m, x + static_cast<size_t>(T - 1) * m->dims.d_model, last_logits, first_token, lm_ws, st);
  return e == cudaSuccess ? QCF_OK : cuda_error(e, "qcf_full_prefill: lm head");
}

size_t qcf_request_workspace_size(const qcf_dims* dims, int C, int Q, int n_anchor_total, int N) {
  if (!dims || C <= 0 || Q <= 0 || N < 0 || N > C || n_anchor_total < 0) return 0;
  // staging holds every chunk's anchors for the probe layers; bound it by the total anchor count
  Carve c{nullptr, 0};
  RequestLayout r;
  const int crit = dims->n_layers;  // upper bound on probe layers
  carve_request(c, *dims, C, Q, n_anchor_total, N, 1, crit, n_anchor_total > 0 ? n_anchor_total : 1, &r);
  return c.used;
}

size_t qcf_request_workspace_size_for(const qcf_dims* dims, const qcf_request* r) {
  if (!dims || !r || !r->chunk_len || r->n_chunks <= 0 || r->n_chunks > kMaxReqChunks || r->query_len <= 0 ||
      r->ratio_bp < 0 || r->ratio_bp > 10000 || r->n_anchor < 0)
    return 0;
  long long Cl = 0;
  for (int c = 0; c < r->n_chunks; ++c) {
    if (r->chunk_len[c] <= 0) return 0;
    Cl += r->chunk_len[c];
  }
  if (Cl > (1 << 30)) return 0;
  const int C = static_cast<int>(Cl), Q = r->query_len, L = dims->n_layers;
  int N = 0;
  qcf_num_selected(C, r->ratio_bp, &N);
  Carve c{nullptr, 0};
  if (r->selector == QCF_SELECT_HKVD) {
    std::vector<int> Nl;
    if (!hkvd_counts(r->layer_ratio_bp, L, C, r->ratio_bp, &Nl)) return 0;
    HkvdLayout H;
    carve_hkvd(c, *dims, C, Q, Nl, &H);
    return c.used;
  }
  const int crit = r->selector == QCF_SELECT_ALL_LAYERS ? L - 1 : r->crit_layer;
  if (crit < 0 || crit >= L) return 0;
  const int nA = crit > 0 ? r->n_anchor * r->n_chunks : 0;
  RequestLayout rl;
  carve_request(c, *dims, C, Q, nA, N, r->n_chunks, crit, r->n_anchor, &rl);
  return c.used;
}

qcf_status qcf_request_prefill(const qcf_model* m, const qcf_request* r, const qcf_outputs* out, void* ws,
                               size_t ws_bytes, void* compute_stream, void* copy_stream) {
  ReqPlan P;
  qcf_status s = request_plan(m, r, out, ws, ws_bytes, &P);
  if (s != QCF_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t xs = static_cast<cudaStream_t>(copy_stream);
  const int L = m->dims.n_layers;
  EventPool& pool = event_pool();
  std::lock_guard<std::mutex> lk(pool.mu);
  cudaEvent_t* ev = nullptr;
  if (!pool.get(static_cast<size_t>(L) + 3, &ev)) return set_error(QCF_ERR_CUDA, "qcf_request_prefill: event create");
  cudaEvent_t ev_start = ev[0], ev_anchor = ev[1], ev_crit = ev[2];
  cudaEvent_t* ev_layer = ev + 3;
  cudaError_t e = cudaEventRecord(ev_start, cs);
  if (e != cudaSuccess) return cuda_error(e, "qcf_request_prefill: record start");
  if ((e = cudaStreamWaitEvent(xs, ev_start, 0)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: copy wait");
  // ---- copy stream: anchors of the probe layers, the critical layer's keys, then every layer in
  // order; the per-layer copies (most of the host's calls) are enqueued after the probe's launches
  if (take_fault(3)) return set_error(QCF_ERR_CUDA, "qcf_request_prefill: injected host-to-device copy failure");
  if ((s = request_copy_anchors(m, r, P, xs)) != QCF_OK) return s;
  if ((e = cudaEventRecord(ev_anchor, xs)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill: record");
  if ((s = request_copy_layers(m, r, out, P, xs, ev_crit, ev_layer, true)) != QCF_OK) return s;
  P.wait_stride = kPinnedWaitStride;
  return request_compute(m, r, out, P, cs, ev_anchor, ev_crit, ev_layer,
                         [&] { return request_copy_layers(m, r, out, P, xs, ev_crit, ev_layer, false); });
}

size_t qcf_storage_staging_bytes(const qcf_dims* dims, const qcf_request* r) {
  if (!dims || !r || !r->chunk_len || r->n_chunks <= 0) return 0;
  int64_t C = 0;
  for (int c = 0; c < r->n_chunks; ++c) {
    if (r->chunk_len[c] <= 0) return 0;
    C += r->chunk_len[c];
  }
  return static_cast<size_t>(4 * C) * dims->n_kv_heads * dims->head_dim * sizeof(qcf_bf16);
}

qcf_status qcf_request_prefill_storage(const qcf_model* m, const qcf_request* r, const qcf_chunk_file* files,
                                       void* staging, size_t staging_bytes, const qcf_outputs* out, void* ws,
                                       size_t ws_bytes, void* compute_stream, void* copy_stream) {
  if (!m || !r || !files || !staging || !r->chunk_len)
    return set_error(QCF_ERR_INVALID_ARG, "qcf_request_prefill_storage: NULL pointer");
  if (r->n_chunks <= 0 || r->n_chunks > kMaxReqChunks)
    return set_error(QCF_ERR_SHAPE, "qcf_request_prefill_storage: n_chunks=%d", r->n_chunks);
  const size_t need = qcf_storage_staging_bytes(&m->dims, r);
  if (need == 0 || staging_bytes < need)
    return set_error(QCF_ERR_WORKSPACE, "qcf_request_prefill_storage: staging %zu < %zu bytes", staging_bytes, need);
  for (int c = 0; c < r->n_chunks; ++c)
    if (files[c].fd < 0 || files[c].k_offset < 0 || files[c].v_offset < 0 || files[c].layer_stride < 0)
      return set_error(QCF_ERR_INVALID_ARG, "qcf_request_prefill_storage: chunk %d file", c);
  // the chunk host pointers are not read on this path: point them at the staging buffer
  // so the shared validation accepts the request
  std::vector<const qcf_bf16*> host_ptrs(r->n_chunks, static_cast<const qcf_bf16*>(staging));
  qcf_request rr = *r;
  rr.chunk_K_host = host_ptrs.data();
  rr.chunk_V_host = host_ptrs.data();
  ReqPlan P;
  qcf_status s = request_plan(m, &rr, out, ws, ws_bytes, &P);
  if (s != QCF_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t xs = static_cast<cudaStream_t>(copy_stream);
  const int L = m->dims.n_layers;
  EventPool& pool = event_pool();
  std::lock_guard<std::mutex> lk(pool.mu);
  cudaEvent_t* ev = nullptr;
  if (!pool.get(static_cast<size_t>(L) + 3, &ev)) return set_error(QCF_ERR_CUDA, "qcf_request_prefill_storage: events");
  cudaEvent_t ev_start = ev[0], ev_anchor = ev[1], ev_crit = ev[2];
  cudaEvent_t* ev_layer = ev + 3;
  cudaError_t e = cudaEventRecord(ev_start, cs);
  if (e != cudaSuccess) return cuda_error(e, "qcf_request_prefill_storage: record start");
  if ((e = cudaStreamWaitEvent(xs, ev_start, 0)) != cudaSuccess)
    return cuda_error(e, "qcf_request_prefill_storage: copy wait");
  if ((s = request_copy_anchors(m, &rr, P, xs)) != QCF_OK) return s;
  if ((e = cudaEventRecord(ev_anchor, xs)) != cudaSuccess) return cuda_error(e, "qcf_request_prefill_storage: record");
  StorageCtx* ctx = new StorageCtx;
  ctx->files.assign(files, files + r->n_chunks);
  ctx->len.assign(r->chunk_len, r->chunk_len + r->n_chunks);
  ctx->row_bytes = static_cast<size_t>(m->dims.n_kv_heads) * m->dims.head_dim * sizeof(qcf_bf16);
  ctx->C = static_cast<size_t>(P.C);
  ctx->buf[0] = static_cast<uint8_t*>(staging);
  ctx->buf[1] = static_cast<uint8_t*>(staging) + 2 * ctx->C * ctx->row_bytes;
  if ((s = request_copy_layers_storage(m, out, P, ctx, xs, ev_crit, ev_layer)) != QCF_OK) return s;
  return request_compute(m, &rr, out, P, cs, ev_anchor, ev_crit, ev_layer);
}

qcf_status qcf_storage_status(int* err) {
  if (!err) return set_error(QCF_ERR_INVALID_ARG, "qcf_storage_status: NULL pointer");
  *err = g_storage_err.exchange(0);
  return QCF_OK;
}

size_t qcf_batch_workspace_size(const qcf_dims* dims, const qcf_request* reqs, int n_req) {
  if (!dims || !reqs || n_req <= 0 || n_req > kMaxBatch) return 0;
  size_t total = 0;
  std::vector<int> Cs;
  for (int i = 0; i < n_req; ++i) {
    const size_t sz = qcf_request_workspace_size_for(dims, &reqs[i]);
    if (!sz) return 0;
    total = align_up(total + sz, 256);
    int C = 0;
    for (int c = 0; c < reqs[i].n_chunks; ++c) C += reqs[i].chunk_len[c];
    Cs.push_back(C);
  }
  UniqueChunks U;
  if (!unique_chunks(reqs, n_req, &U)) return 0;
  Carve c{nullptr, 0};
  BatchStaging B;
  carve_staging(c, *dims, U, Cs, &B);
  std::vector<MergedProbe> groups = merged_probe_groups(*dims, reqs, n_req);
  for (MergedProbe& g : groups) carve_merged_probe(c, *dims, &g);
  return total + c.used + 256;
}

qcf_status qcf_batch_prefill(const qcf_model* m, const qcf_request* reqs, const qcf_outputs* outs, int n_req,
                             void* ws, size_t ws_bytes, void* compute_stream, void* copy_stream, int64_t* h2d_bytes) {
  if (!m || !reqs || !outs || !ws) return set_error(QCF_ERR_INVALID_ARG, "qcf_batch_prefill: NULL pointer");
  if (n_req <= 0 || n_req > kMaxBatch) return set_error(QCF_ERR_SHAPE, "qcf_batch_prefill: n_req=%d not in [1,%d]", n_req, kMaxBatch);
  if (!aligned16(ws)) return set_error(QCF_ERR_ALIGN, "qcf_batch_prefill: workspace misaligned");
  const qcf_dims& d = m->dims;
  const int L = d.n_layers;
  std::vector<ReqPlan> P(n_req);
  std::vector<int> Cs;
  size_t off = 0;
  for (int i = 0; i < n_req; ++i) {
    if (off > ws_bytes) return set_error(QCF_ERR_WORKSPACE, "qcf_batch_prefill: workspace too small");
    qcf_status s = request_plan(m, &reqs[i], &outs[i], static_cast<uint8_t*>(ws) + off, ws_bytes - off, &P[i]);
    if (s != QCF_OK) return s;
    off = align_up(off + P[i].ws_used, 256);
    Cs.push_back(P[i].C);
  }
  UniqueChunks U;
  if (!unique_chunks(reqs, n_req, &U)) return set_error(QCF_ERR_INVALID_ARG, "qcf_batch_prefill: chunk tables");
  if (off > ws_bytes) return set_error(QCF_ERR_WORKSPACE, "qcf_batch_prefill: workspace too small");
  Carve cv{static_cast<uint8_t*>(ws) + off, ws_bytes - off};
  BatchStaging B;
  if (!carve_staging(cv, d, U, Cs, &B)) return set_error(QCF_ERR_WORKSPACE, "qcf_batch_prefill: workspace too small");
  std::vector<MergedProbe> groups = merged_probe_groups(d, reqs, n_req);
  std::vector<char> probe_done(n_req, 0);
  for (MergedProbe& g : groups) {
    if (!carve_merged_probe(cv, d, &g)) return set_error(QCF_ERR_WORKSPACE, "qcf_batch_prefill: workspace too small");
    for (int i : g.members) probe_done[i] = 1;
  }
  // row maps: request row -> staging row, and the rotation offset of its chunk in this request
  std::vector<std::vector<int32_t>> src_row(n_req), delta(n_req);
  for (int i = 0; i < n_req; ++i) {
    src_row[i].resize(P[i].C);
    delta[i].resize(P[i].C);
    for (int c = 0; c < reqs[i].n_chunks; ++c) {
      const int u = U.of_req[i][c], o = P[i].seg_start[c];
      for (int j = 0; j < reqs[i].chunk_len[c]; ++j) {
        src_row[i][o + j] = U.start[u] + j;
        delta[i][o + j] = o;
      }
    }
  }
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t xs = static_cast<cudaStream_t>(copy_stream);
  const size_t HD = static_cast<size_t>(d.n_kv_heads) * d.head_dim;
  const size_t eb = sizeof(qcf_bf16);
  // events: start and anchors shared; each request has its own critical-layer and per-layer
  // events, recorded right after its own cache rows are written, so a request never waits
  // for another request's copies
  EventPool& pool = event_pool();
  std::lock_guard<std::mutex> lk(pool.mu);
  cudaEvent_t* ev = nullptr;
  const size_t per_req_ev = static_cast<size_t>(L) + 1;
  if (!pool.get(2 + n_req * per_req_ev, &ev)) return set_error(QCF_ERR_CUDA, "qcf_batch_prefill: event create");
  cudaEvent_t ev_start = ev[0], ev_anchor = ev[1];
  auto ev_crit_of = [&](int i) { return ev[2 + i * per_req_ev]; };
  auto ev_layer_of = [&](int i) { return ev + 2 + i * per_req_ev + 1; };
  cudaError_t e = cudaEventRecord(ev_start, cs);
  if (e != cudaSuccess) return cuda_error(e, "qcf_batch_prefill: record start");
  if ((e = cudaStreamWaitEvent(xs, ev_start, 0)) != cudaSuccess) return cuda_error(e, "qcf_batch_prefill: copy wait");
  int64_t h2d = 0;
  for (int i = 0; i < n_req; ++i) {
    if ((e = cudaMemcpyAsync(B.src_row[i], src_row[i].data(), P[i].C * sizeof(int32_t), cudaMemcpyHostToDevice, xs)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(B.delta[i], delta[i].data(), P[i].C * sizeof(int32_t), cudaMemcpyHostToDevice, xs)) !=
            cudaSuccess)
      return cuda_error(e, "qcf_batch_prefill: row maps");
    h2d += 2 * static_cast<int64_t>(P[i].C) * sizeof(int32_t);
  }
  // anchors: per request (each request's probe reads its own staging)
  for (int i = 0; i < n_req; ++i) {
    qcf_status s = request_copy_anchors(m, &reqs[i], P[i], xs);
    if (s != QCF_OK) return s;
    h2d += static_cast<int64_t>(P[i].nA > 0 ? reqs[i].n_chunks : 0) * P[i].crit * P[i].A * HD * eb * 2;
  }
  if ((e = cudaEventRecord(ev_anchor, xs)) != cudaSuccess) return cuda_error(e, "qcf_batch_prefill: record");
  // every distinct chunk crosses the host link once per layer (and once more for a critical layer)
  auto stage = [&](int l, __nv_bfloat16* dK, __nv_bfloat16* dV) -> cudaError_t {
    for (size_t u = 0; u < U.K.size(); ++u) {
      const size_t n_el = static_cast<size_t>(U.len[u]) * HD;
      const size_t src = static_cast<size_t>(l) * n_el, dst = static_cast<size_t>(U.start[u]) * HD;
      cudaError_t ce;
      if (dK && (ce = cudaMemcpyAsync(dK + dst, U.K[u] + src, n_el * eb, cudaMemcpyHostToDevice, xs)) != cudaSuccess)
        return ce;
      if (dV && (ce = cudaMemcpyAsync(dV + dst, U.V[u] + src, n_el * eb, cudaMemcpyHostToDevice, xs)) != cudaSuccess)
        return ce;
      h2d += static_cast<int64_t>(n_el * eb) * ((dK ? 1 : 0) + (dV ? 1 : 0));
    }
    return cudaSuccess;
  };
  std::vector<int> crits;
  for (int i = 0; i < n_req; ++i)
    if (std::find(crits.begin(), crits.end(), P[i].crit) == crits.end()) crits.push_back(P[i].crit);
  for (int c : crits) {
    if ((e = stage(c, B.Kc, nullptr)) != cudaSuccess) return cuda_error(e, "qcf_batch_prefill: critical-layer copy");
    for (int i = 0; i < n_req; ++i) {
      if (P[i].crit != c) continue;
      if ((e = launch_stage_scatter(B.Kc, nullptr, B.src_row[i], B.delta[i], P[i].C, U.rows, d.n_kv_heads, d.head_dim,
                                    &m->rope, reinterpret_cast<__nv_bfloat16*>(outs[i].K_layers[c]), nullptr, true,
                                    false, xs)) != cudaSuccess)
        return cuda_error(e, "qcf_batch_prefill: scatter");
      if ((e = cudaEventRecord(ev_crit_of(i), xs)) != cudaSuccess) return cuda_error(e, "qcf_batch_prefill: record");
    }
  }
  // the per-layer staging copies (most of the host's calls) are enqueued after the first
  // request's probe launches, as for a single request
  auto enqueue_layers = [&]() -> qcf_status {
    for (int l = 0; l < L; ++l) {
      bool need_k = false;
      for (int i = 0; i < n_req; ++i) need_k |= P[i].crit != l;
      const int b = l & 1;
      if ((e = stage(l, need_k ? B.K[b] : nullptr, B.V[b])) != cudaSuccess)
        return cuda_error(e, "qcf_batch_prefill: layer copy");
      for (int i = 0; i < n_req; ++i) {
        if ((e = launch_stage_scatter(B.K[b], B.V[b], B.src_row[i], B.delta[i], P[i].C, U.rows, d.n_kv_heads,
                                      d.head_dim, &m->rope, reinterpret_cast<__nv_bfloat16*>(outs[i].K_layers[l]),
                                      reinterpret_cast<__nv_bfloat16*>(outs[i].V_layers[l]), P[i].crit != l, true,
                                      xs)) != cudaSuccess)
          return cuda_error(e, "qcf_batch_prefill: scatter");
        if ((e = cudaEventRecord(ev_layer_of(i)[l], xs)) != cudaSuccess) return cuda_error(e, "qcf_batch_prefill: record");
      }
    }
    if (h2d_bytes) *h2d_bytes = h2d;
    return QCF_OK;
  };
  // compute: the merged probes, then the requests one after another, each waiting only for
  // the layers it reaches
  for (MergedProbe& g : groups) {
    qcf_status s = run_merged_probe(m, reqs, P, g, cs, ev_anchor);
    if (s != QCF_OK) return s;
  }
  for (int i = 0; i < n_req; ++i) {
    P[i].wait_stride = kPinnedWaitStride;
    qcf_status s = request_compute(m, &reqs[i], &outs[i], P[i], cs, ev_anchor, ev_crit_of(i), ev_layer_of(i),
                                   i == 0 ? std::function<qcf_status()>(enqueue_layers) : std::function<qcf_status()>(),
                                   probe_done[i] != 0);
    if (s != QCF_OK) return s;
  }
  return QCF_OK;
}

}  // extern "C"
