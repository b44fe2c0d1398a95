/*
 * qcf.h -- C ABI of a GB300 (sm_103a) library for query-centric KV-cache fusion
 * in retrieval-augmented prefill.
 *
 * The method (QCFuse: Query-Centric Cache Fusion for Efficient RAG Inference,
 * technical summary, section 2 "Methodology"; CacheBlend's selective recompute
 * as described in "KVCache reuse 01", section 1.3):
 *   offline  each retrieved chunk is prefilled alone at positions 0..L-1 and its
 *            per-layer K/V kept in host memory; a few tokens of largest key norm
 *            per chunk are kept as anchors;
 *   online   the query runs the first layers with the anchors as a KV prefix,
 *            one critical middle layer's keys are scored by the query's softmax
 *            attention mass, the top-N context tokens are selected, and layer by
 *            layer only those rows (plus the query) are recomputed, attending to
 *            the fused cache with causality by true position, while the next
 *            layer's chunk K/V streams in from host memory.
 *
 * Conventions (every entry point):
 *  - Returns qcf_status.  Argument errors are reported synchronously before any
 *    launch; the message of the last error on the calling thread is returned by
 *    qcf_last_error().  No C++ exception crosses this boundary.
 *  - Pointers are device memory owned by the caller unless documented as host
 *    (pageable or pinned).  The library never allocates device memory on these
 *    paths and never frees caller memory.  Scratch comes from the caller as
 *    (ws, ws_bytes), sized by the matching *_workspace_size() function, 256-byte
 *    aligned; too small gives QCF_ERR_WORKSPACE.
 *  - Work is enqueued asynchronously on the caller's CUDA stream, passed as
 *    void* (a cudaStream_t; NULL is the legacy default stream).
 *  - Device-side failures (a bounded wait that ran out, an index that failed a
 *    check) set bits of a device status word instead of trapping; read and clear
 *    it with qcf_query_status() after synchronising.
 *  - Tensors are row-major and contiguous: K/V caches are [rows][H_kv][D], query
 *    blocks [rows][H_q][D], hidden states [rows][d].  bf16 buffers are passed as
 *    qcf_bf16 (the raw 16-bit pattern).  Base pointers must be 16-byte aligned
 *    (QCF_ERR_ALIGN otherwise).
 *  - Supported head dims D: 16, 64, 128.  H_q must be a multiple of H_kv.
 *  - Indices and positions are int32; position tables are strictly ascending.
 */
#ifndef QCF_H_
#define QCF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t qcf_bf16;

typedef enum qcf_status {
  QCF_OK = 0,
  QCF_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum */
  QCF_ERR_SHAPE = 2,        /* sizes inconsistent or outside the supported set */
  QCF_ERR_ALIGN = 3,        /* pointer or stride not 16-byte aligned */
  QCF_ERR_WORKSPACE = 4,    /* ws_bytes smaller than the *_workspace_size() */
  QCF_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
  QCF_ERR_TIMEOUT = 6,      /* a device-side bounded wait ran out */
  QCF_ERR_UNSUPPORTED = 7,  /* no sm_103a device, or a feature not built */
  QCF_ERR_DEVICE = 8        /* a device-side index check failed */
} qcf_status;

/* Device status word bits (qcf_query_status). */
#define QCF_DEV_TIMEOUT 0x1u
#define QCF_DEV_BAD_INDEX 0x2u

/* ------------------------------------------------------------------ library */

/* Message of the last error on this thread ("" when none). Never NULL. */
const char* qcf_last_error(void);
/* Version string of the library build. */
const char* qcf_version(void);
/* Reads and clears the device status word (bits QCF_DEV_*), synchronising
 * `stream` first.  *status = 0 means no device-side failure was seen. */
qcf_status qcf_query_status(void* stream, uint32_t* status);
/* Host-side fault injection for tests: the next call of the given kind fails
 * before launching anything.  0 clears.  Kinds: 1 = invalid index table,
 * 2 = short workspace, 3 = failed host-to-device copy, 4 = misaligned pointer. */
qcf_status qcf_debug_set_fault(int kind);
/* Enables device-side index checks (positions ascending and in range) in the
 * kernels that read index tables; failures set QCF_DEV_BAD_INDEX. */
qcf_status qcf_set_check(int on);
/* Total kernel launches issued by the library since load (all entry points). */
int64_t qcf_launch_count(void);

/* Per-kernel timing with CUDA events recorded around each launch on the
 * launching stream.  Enable, run, then read: names/ms/launches of up to `max`
 * kernel classes; reading synchronises on the recorded events and resets. */
qcf_status qcf_timing_enable(int on);
qcf_status qcf_timing_read(int max, const char** names, double* ms, int64_t* launches, int* n_classes);

/* Measures the special-function unit's exp2 throughput of the current device (exp2 per
 * second over all SMs): eight independent chains of ex2.approx per thread, the best of
 * two timed launches after one warm-up.  The ceiling of the critical-layer profile, which
 * evaluates two exponentials per score-row element.  scratch: device memory of at least
 * num_SMs * 8 * 256 * 4 bytes (the kernel's outputs).  Synchronises the stream. */
qcf_status qcf_calibrate_exp2_rate(float* scratch, size_t scratch_bytes, double* per_second, void* stream);

/* ------------------------------------------------------------------ shapes */

/* N = ceil(ratio * C) for a recompute ratio in basis points (1500 = 15 %),
 * computed in integers and clamped to [0, C]: the number of context tokens
 * recomputed (Cache-Craft's N = ceil(CFO * |C_i|), "KVCache reuse 01" 2.3.3). */
qcf_status qcf_num_selected(int C, int ratio_bp, int* N);

/* RoPE tables, rotate-half convention: pair (k, k + D/2) of a head at position p
 * turns by angle p * theta^(-2k/D).  cos/sin are device [max_pos][D/2] fp32. */
typedef struct qcf_rope_table {
  const float* cos;
  const float* sin;
  int max_pos;
  int head_dim;
} qcf_rope_table;

/* Fills host buffers cos_host/sin_host [max_pos][D/2] with the angles taken in
 * fp64 and rounded to fp32 (the caller copies them to the device). */
qcf_status qcf_rope_table_fill_host(float* cos_host, float* sin_host, int max_pos, int D, double theta);

/* ------------------------------------------------------------------ offline */

/* Semantic-summary anchors (QCFuse 2.A "Anchor-based Lightweight Query
 * Probing"): for each chunk, the n_anchor tokens whose key has the largest L2
 * norm over all H_kv*D entries, ties to the lower index, written ascending and
 * chunk-local to anchor_idx [n_chunks][n_anchor].
 *   K            device [C][Hkv][D] bf16, the critical layer's stored keys
 *   chunk_start  HOST [n_chunks + 1], ascending, chunk_start[n_chunks] = C;
 *                every chunk needs length >= n_anchor and <= 16384
 *   norms        device [C] fp32 key norms, or NULL
 * Norms are accumulated in fp32. */
qcf_status qcf_anchor_keynorm_topk(const qcf_bf16* K, const int32_t* chunk_start, int n_chunks,
                                   int Hkv, int D, int n_anchor, int32_t* anchor_idx, float* norms,
                                   void* stream);

/* ------------------------------------------------------------------ online steps */

/* Re-rotation of reused keys to their new absolute positions ("adjust the
 * positional encoding" of chunks not at the prefix, CacheBlend problem
 * definition 2.4): row i of segment s becomes R(delta[s]) * K_src[i].
 *   K_src, K_dst  device [n_rows][Hkv][D] bf16; may be the same buffer (in place)
 *   seg_start     HOST [n_seg + 1] ascending, seg_start[n_seg] = n_rows
 *   seg_delta     HOST [n_seg], 0 <= delta < t->max_pos
 * Rotation in fp32 from the fp32 table, rounded to bf16. */
qcf_status qcf_rope_reposition(const qcf_bf16* K_src, qcf_bf16* K_dst, int64_t n_rows, int Hkv, int D,
                               const int32_t* seg_start, const int32_t* seg_delta, int n_seg,
                               const qcf_rope_table* t, void* stream);

/* Critical-layer attention profiling (QCFuse 2.A "Critical-layer Attention
 * Profiling"): score[j] = sum over query rows r and heads h of
 * softmax_j(scale * q[r,h] . K[j, h / (Hq/Hkv)]) over the C context keys.
 *   q       device [nq][Hq][D] bf16
 *   K       device [C][Hkv][D] bf16 (already re-rotated)
 *   scores  device [C] fp32
 * Products on tensor cores (fp32 accumulate), softmax in fp32 with exact
 * per-row max and normaliser (two passes over K). */
size_t qcf_profile_scores_workspace_size(int nq, int C, int Hq, int Hkv, int D);
qcf_status qcf_profile_scores(const qcf_bf16* q, const qcf_bf16* K, int nq, int C, int Hq, int Hkv, int D,
                              float scale, float* scores, void* ws, size_t ws_bytes, void* stream);

/* qcf_profile_scores with no caller workspace and no allocation of any kind.
 * The pages have no counterpart: this exists for callers that cannot allocate
 * device memory at the point of the call -- for example a serving loop that
 * gave all free device memory to its KV-cache pool at start-up, or code holding
 * a memory budget fixed in advance that must not call cudaMalloc (which may
 * also synchronise the device) on the request path.
 * Scratch is one fixed 8 MiB array in device global memory, present on every
 * GPU that loads the library for the life of the process.  A shape whose
 * qcf_profile_scores_workspace_size() exceeds 8 MiB is rejected with
 * QCF_ERR_WORKSPACE before anything runs; the 8B-shaped request (64 query rows
 * x 32 heads over 5120 keys) needs under 1 MiB and 131072 keys under 6 MiB.
 * The first call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All calls
 * share the one array: calls that overlap on the GPU (different streams, or
 * host threads without ordering) race and corrupt each other's results.  Every
 * call rewrites all the scratch it reads, so no clearing is needed.
 * Arguments, layouts and results are those of qcf_profile_scores. */
qcf_status qcf_profile_scores_noalloc(const qcf_bf16* q, const qcf_bf16* K, int nq, int C, int Hq, int Hkv, int D,
                                      float scale, float* scores, void* stream);

/* Top-N selection (QCFuse 2.A: "the Top-N context token indices"): the indices of
 * the N largest scores, ties to the lower index (the order of a stable sort by
 * descending score), written ascending to sel [N].  0 <= N <= C <= 2^24.
 * Exact on the fp32 bit patterns; -0.0 counts as +0.0; scores must not be NaN. */
qcf_status qcf_topn_select(const float* scores, int C, int N, int32_t* sel, void* stream);

/* Top-N selection with scratch, for long score vectors: the same result as
 * qcf_topn_select.  Above 16384 scores the work spreads over a cooperative grid of
 * up to one CTA per SM (4096 scores each) that reads the scores once and meets at
 * bounded grid barriers (a barrier that runs out sets QCF_DEV_TIMEOUT and leaves sel
 * incomplete); at or below 16384 scores, or beyond what one resident grid covers,
 * this is qcf_topn_select and ws is not touched.
 *   ws  device scratch of qcf_topn_select_workspace_size(C) bytes (0 for C <= 16384,
 *       then ws may be NULL); it needs no clearing (each call resets the state it
 *       uses, on the GPU); calls that overlap on the GPU need separate scratch. */
size_t qcf_topn_select_workspace_size(int C);
qcf_status qcf_topn_select_ws(const float* scores, int C, int N, int32_t* sel, void* ws, size_t ws_bytes,
                              void* stream);

/* KV deviation of recomputed rows ("KVCache reuse 01" 1.3.2, "KV Deviation"): for i < n,
 * dev[i] = sum over the Hkv*D entries of (k_new[i] - K_cache[pos[i]])^2 + (v_new[i] - V_cache[pos[i]])^2,
 * fp32 accumulation of bf16 inputs.
 *   k_new, v_new  device [n][Hkv][D] bf16 (fresh rows); pos device [n] in [0, T)
 *   K_cache, V_cache device [T][Hkv][D] bf16 (the reused rows); dev device [n] fp32.
 * A position outside [0, T) gives dev 0 and sets QCF_DEV_BAD_INDEX in the device status word. */
qcf_status qcf_kv_deviation(const qcf_bf16* k_new, const qcf_bf16* v_new, const int32_t* pos, int n,
                            const qcf_bf16* K_cache, const qcf_bf16* V_cache, int T, int Hkv, int D, float* dev,
                            void* stream);

/* Gathers the rows of the tokens chosen for recompute ("KVCache reuse 01" 1.3.4,
 * selective recompute flow: the selected tokens are masked out of the full
 * input and only they run through the layer): dst[i][:] = src[idx[i]][:] for i < n.
 *   src  device [src_rows][width] bf16 (width % 8 == 0); dst device [n][width] bf16
 *   idx  device [n], each in [0, src_rows); an index outside that range is not read:
 *        its dst row is left as it was and QCF_DEV_BAD_INDEX is set in the status word. */
qcf_status qcf_gather_rows(const qcf_bf16* src, int64_t src_rows, int width, const int32_t* idx, int n,
                           qcf_bf16* dst, void* stream);

/* Writes fresh K/V rows of the recomputed tokens into the fused cache at their
 * positions ("KVCache reuse 01" 1.3.4: the recomputed K_i, V_i extend the reused
 * cache, and attention then runs over all tokens of the layer):
 * K_cache[pos[i]] = k_new[i], V_cache[pos[i]] = v_new[i].
 *   k_new, v_new  device [n][Hkv][D] bf16; pos device [n] in [0, T), distinct. */
qcf_status qcf_scatter_kv(const qcf_bf16* k_new, const qcf_bf16* v_new, const int32_t* pos, int n, int Hkv,
                          int D, qcf_bf16* K_cache, qcf_bf16* V_cache, int T, void* stream);

/* Location-aware sparse causal attention (QCFuse 2.A: a discrete token index
 * table, causal constraint by true position): for each recomputed row i at
 * position pos[i], o[i,h] = sum_{j <= pos[i]} softmax_j(scale * q[i,h] . K[j,g]) V[j,g]
 * with g = h / (Hq/Hkv), over the fused cache (reused rows plus fresh rows).
 *   q    device [n][Hq][D] bf16;  pos device [n] strictly ascending, < T
 *   K,V  device [T][Hkv][D] bf16; o device [n][Hq][D] bf16
 *   lse  device [n][Hq] fp32 natural-log sum of exp of the scaled logits, or NULL
 * Tensor-core QK^T and PV (fp32 accumulate), online softmax in fp32. */
size_t qcf_sparse_causal_attn_workspace_size(int n, int T, int Hq, int Hkv, int D);
qcf_status qcf_sparse_causal_attn(const qcf_bf16* q, const int32_t* pos, int n, const qcf_bf16* K,
                                  const qcf_bf16* V, int T, int Hq, int Hkv, int D, float scale, qcf_bf16* o,
                                  float* lse, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ dense pieces */

/* out = A * W^T for A device [M][K] bf16 and W device [N][K] bf16 (nn.Linear
 * layout) on tcgen05 tensor cores with TMEM accumulators.
 *   epilogue QCF_EPI_STORE_BF16: out is bf16 [M][N]
 *   epilogue QCF_EPI_ADD_F32:    out is fp32 [M][N] and receives out += A W^T
 *   | QCF_LINEAR_W_KN:           W is stored [K][N] instead (out = A * W)
 * K % 64 == 0, N % 64 == 0.  ws: device scratch of qcf_linear_workspace_size
 * bytes (tile counters and fp32 partial sums when the planner shares output
 * tiles between CTAs); its contents need not survive between calls, but calls
 * that share it must be ordered on one stream.  Results are bitwise repeatable
 * for the same inputs and shapes (partial sums are added in a fixed order). */
#define QCF_EPI_STORE_BF16 0
#define QCF_EPI_ADD_F32 1
#define QCF_LINEAR_W_KN 0x10
size_t qcf_linear_workspace_size(int M, int N, int K);
qcf_status qcf_linear(const qcf_bf16* A, int M, int K, const qcf_bf16* W, int N, int epilogue, void* out,
                      void* ws, size_t ws_bytes, void* stream);

/* h = x / sqrt(mean(x^2) + eps) * g per row; x device fp32 [n][d], g bf16 [d],
 * h bf16 [n][d].  Statistics in fp32. */
qcf_status qcf_rmsnorm(const float* x, int n, int d, const qcf_bf16* g, float eps, qcf_bf16* h, void* stream);

/* ------------------------------------------------------------------ model */

typedef struct qcf_dims {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim;
  int ffn;         /* FFN width of the model */
  int ffn_padded;  /* ffn rounded up to a multiple of 64 (zero rows/columns) */
  int vocab;
  float eps;
  float theta;
} qcf_dims;

/* One decoder layer's weights, device bf16, packed for the tensor-core GEMMs:
 *   w_qkv   [(Hq + 2 Hkv) D][d]   rows W_q, then W_k, then W_v
 *   w_o     [d][Hq D]
 *   w_gu    [2 ffn_padded][d]     blocks of 64 gate rows then the same 64 up rows
 *   w_down  [d][ffn_padded]       columns beyond ffn are zero
 *   g_attn, g_mlp [d]             RMSNorm gains */
typedef struct qcf_layer_weights {
  const qcf_bf16* w_qkv;
  const qcf_bf16* w_o;
  const qcf_bf16* w_gu;
  const qcf_bf16* w_down;
  const qcf_bf16* g_attn;
  const qcf_bf16* g_mlp;
} qcf_layer_weights;

typedef struct qcf_model {
  qcf_dims dims;
  const qcf_bf16* embed;            /* device [vocab][d] */
  const qcf_bf16* lm_head;          /* device [vocab][d] */
  const qcf_bf16* g_final;          /* device [d] */
  const qcf_layer_weights* layers;  /* HOST array [n_layers] */
  qcf_rope_table rope;              /* max_pos must exceed every position used */
} qcf_model;

/* One decoder layer for n recomputed rows (the selective recompute flow of
 * "KVCache reuse 01" 1.3.4): RMSNorm -> QKV GEMM with RoPE at rope_pos and the
 * fresh K/V written into the cache at cache_row (before attention) -> sparse
 * causal attention of row i over cache rows <= cache_row[i] -> O GEMM added to
 * x -> RMSNorm -> gate/up GEMM with SwiGLU -> down GEMM added to x.
 *   x          device fp32 [n][d], the residual stream, updated in place
 *   rope_pos   device [n] absolute positions (RoPE phase)
 *   cache_row  device [n] strictly ascending rows of the cache written and used
 *              as each row's causal bound (equal to rope_pos on the fused path)
 *   K_cache, V_cache device [T][Hkv][D] bf16 */
size_t qcf_layer_workspace_size(const qcf_dims* dims, int n, int T);
qcf_status qcf_fused_layer_forward(const qcf_model* m, int layer, float* x, const int32_t* rope_pos,
                                   const int32_t* cache_row, int n, qcf_bf16* K_cache, qcf_bf16* V_cache,
                                   int T, void* ws, size_t ws_bytes, void* stream);

/* Full recompute of T tokens at positions 0..T-1 ("Full KV Recompute",
 * CacheBlend problem definition 2.2): per-layer K/V into K_layers[l]/V_layers[l]
 * (HOST arrays of n_layers device pointers, each [T][Hkv][D]), the last row's
 * logits (device fp32 [vocab]) and the first token (device int32, argmax with
 * the lowest index on ties).  ids device [T]. */
size_t qcf_full_prefill_workspace_size(const qcf_dims* dims, int T);
qcf_status qcf_full_prefill(const qcf_model* m, const int32_t* ids, int T, qcf_bf16* const* K_layers,
                            qcf_bf16* const* V_layers, float* last_logits, int32_t* first_token, void* ws,
                            size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ request driver */

/* A request: retrieved chunks in retrieval order, then the query.
 *   chunk_len       HOST [n_chunks]
 *   chunk_K/V_host  HOST arrays [n_chunks] of PINNED host pointers, each
 *                   [n_layers][chunk_len][Hkv][D] bf16 (post-RoPE at local positions)
 *   anchor_idx      HOST [n_chunks][n_anchor] chunk-local ascending
 *   anchor_K/V_host HOST arrays [n_chunks] of PINNED host pointers, each
 *                   [n_layers][n_anchor][Hkv][D] bf16 (the anchors' stored rows)
 *   ids             device [C + query_len]: chunk tokens in order, then the query
 *   forced_sel      device [N] ascending, or NULL to select by profiling */
typedef struct qcf_request {
  int n_chunks;
  const int32_t* chunk_len;
  const qcf_bf16* const* chunk_K_host;
  const qcf_bf16* const* chunk_V_host;
  int n_anchor;
  const int32_t* anchor_idx;
  const qcf_bf16* const* anchor_K_host;
  const qcf_bf16* const* anchor_V_host;
  const int32_t* ids;
  int query_len;
  int crit_layer;
  int ratio_bp;
  const int32_t* forced_sel;
  /* Appended fields: a zero-initialised request keeps the critical-layer selector. */
  int selector;                  /* QCF_SELECT_*; see below */
  const int32_t* layer_ratio_bp; /* HOST [L], QCF_SELECT_HKVD only: share of C kept after layer l, basis points,
                                    non-increasing, layer_ratio_bp[L-1] == ratio_bp */
} qcf_request;

/* Selectors (qcf_request.selector):
 *   QCF_SELECT_CRITICAL    QCFuse: probe layers 0..crit-1 with the anchor prefix, profile at crit_layer
 *                          (QCFuse 2.A); crit_layer = L-1 is the QCLast variant (QCFuse 4, "Results").
 *   QCF_SELECT_ALL_LAYERS  QCAll (QCFuse 4): the probe runs layers 0..L-2 (anchor stores must hold those
 *                          layers); the profile scores of every layer's query against that layer's
 *                          re-rotated keys are summed, then one top-N selection.  Every layer's keys must
 *                          land before the recompute starts: the cost the pages attribute to all-layer
 *                          profiling.  crit_layer still names the anchors' layer (chosen offline).
 *   QCF_SELECT_HKVD        CacheBlend's KV-deviation selection with gradual filtering ("KVCache reuse 01"
 *                          1.3.2-1.3.4): layer 0 projects K/V for every context token, layer l for the
 *                          tokens kept after layer l-1; a token's deviation is the squared L2 distance of
 *                          its fresh K and V to the reused (re-rotated) cache rows; the top
 *                          ceil(layer_ratio_bp[l] * C / 10000) by deviation (ties to the lower position)
 *                          are kept and get fresh K/V, attention and MLP at layer l with the query rows.
 *                          Anchors, crit_layer and forced_sel are ignored; out->scores gets layer 0's
 *                          deviation of every context token, out->sel the rows kept after the last layer. */
#define QCF_SELECT_CRITICAL 0
#define QCF_SELECT_ALL_LAYERS 1
#define QCF_SELECT_HKVD 2

/* Outputs: the fused cache of every layer (HOST arrays of device pointers
 * [C + Q][Hkv][D]), sel [N], scores [C], q_crit [Q][Hq][D] (nullable), the last
 * query row's logits [vocab], the first token on the device and, when
 * first_token_host (PINNED) is set, copied to the host on compute_stream. */
typedef struct qcf_outputs {
  qcf_bf16* const* K_layers;
  qcf_bf16* const* V_layers;
  int32_t* sel;
  float* scores;
  qcf_bf16* q_crit;
  float* last_logits;
  int32_t* first_token;
  int32_t* first_token_host;
  float* x_rows;  /* device fp32 [N + Q][d] final hidden states of the recomputed rows, or NULL */
  /* Appended: QCF_SELECT_HKVD only, or NULL.  device [L][N_0]: row l holds the N_l context rows kept
   * after layer l (ascending), N_l = ceil(layer_ratio_bp[l] * C / 10000). */
  int32_t* layer_sel;
} qcf_outputs;

/* The per-request fused prefill with the per-layer pipeline (QCFuse 2.A
 * "pipelined cache reconstruction"; the load/recompute pipeline of "KVCache
 * reuse 01" 1.3.5): anchors and the critical layer's keys are copied first, the
 * probe, profiling and top-N run, then layer l is recomputed on compute_stream
 * while later layers' chunk K/V are copied on copy_stream.  Enqueues only. */
size_t qcf_request_workspace_size(const qcf_dims* dims, int C, int Q, int n_anchor_total, int N);
/* Workspace for this particular request, any selector (QCF_SELECT_HKVD needs full-row buffers for
 * layer 0, which the size above does not cover).  0 when the request is malformed. */
size_t qcf_request_workspace_size_for(const qcf_dims* dims, const qcf_request* r);
qcf_status qcf_request_prefill(const qcf_model* m, const qcf_request* r, const qcf_outputs* out, void* ws,
                               size_t ws_bytes, void* compute_stream, void* copy_stream);

/* Storage tier (QCFuse 2.A: chunk KV kept on SSD, layer i+1 loaded while layer i is
 * recomputed; anchors stay in CPU memory).  qcf_request_prefill with the chunks' K/V read
 * from files instead of pinned host arrays (r->chunk_K_host / chunk_V_host are ignored;
 * the anchor stores are still host memory).  Per layer, a host function on the copy stream
 * reads that layer's keys and values of every chunk into one half of `staging` (pinned
 * host memory of qcf_storage_staging_bytes, page-aligned for files opened with O_DIRECT),
 * and the copy stream then copies them into the fused cache and re-rotates the keys; the
 * critical layer's keys are read first.  The read of layer l+2 reuses the half of layer l
 * after its copies completed, so reading overlaps the recompute of the layers already
 * landed, as in qcf_request_prefill.
 *   files[c]  chunk c's file: fd open for reading (not closed by the library); the keys of
 *             layer l, [len][Hkv][D] bf16, at k_offset + l * layer_stride, the values at
 *             v_offset + l * layer_stride.  With O_DIRECT, offsets and block sizes must
 *             meet the file system's alignment.
 * A failed or short read leaves that layer's rows undefined (no device fault) and is
 * reported, once the copy stream has run past it, by qcf_storage_status (the first
 * failure's errno since the last call, then cleared; 0 when none). */
typedef struct qcf_chunk_file {
  int fd;
  int64_t k_offset;
  int64_t v_offset;
  int64_t layer_stride;
} qcf_chunk_file;
size_t qcf_storage_staging_bytes(const qcf_dims* dims, const qcf_request* r);
qcf_status qcf_request_prefill_storage(const qcf_model* m, const qcf_request* r, const qcf_chunk_file* files,
                                       void* staging, size_t staging_bytes, const qcf_outputs* out, void* ws,
                                       size_t ws_bytes, void* compute_stream, void* copy_stream);
qcf_status qcf_storage_status(int* err);

/* Several requests whose retrieved chunks overlap (QCFuse 1: retrieved context chunks of
 * different queries overlap by more than 70 %; 2.B: a position-independent cache index
 * with content-based hash search).  A chunk is the same chunk when two requests pass the
 * same host K and V arrays with the same length (a content-keyed chunk store gives equal
 * chunks the same arrays).  On copy_stream every distinct chunk's K and V of a layer
 * cross the host link once, into a shared staging area, and are written from there into
 * each request's fused cache with that request's own offset (keys re-rotated, values
 * copied).  On compute_stream, consecutive requests with the same critical layer
 * (critical-layer selector, head dim 128, at most 128 query rows together once each
 * request's are rounded up to the attention row block) run their probe as one: each
 * probe layer's weights stream once for the group, each request attending only to its
 * own anchors and query rows; then every request runs its profile, selection and
 * recompute as qcf_request_prefill would, waiting only for the layers it reaches.
 * Results are bitwise those of qcf_request_prefill per request.
 *   reqs, outs   host arrays [n_req], 1 <= n_req <= 64, any selectors
 *   ws           device, qcf_batch_workspace_size(dims, reqs, n_req) bytes, caller-owned
 *   h2d_bytes    host, nullable: bytes this call sends host -> device
 * Enqueues only; argument errors are returned before any launch. */
size_t qcf_batch_workspace_size(const qcf_dims* dims, const qcf_request* reqs, int n_req);
qcf_status qcf_batch_prefill(const qcf_model* m, const qcf_request* reqs, const qcf_outputs* outs, int n_req,
                             void* ws, size_t ws_bytes, void* compute_stream, void* copy_stream, int64_t* h2d_bytes);

/* Embedding rows as fp32 residual: x[i] = embed[ids[rows[i]]] (device). */
qcf_status qcf_embed_rows(const qcf_model* m, const int32_t* ids, const int32_t* rows, int n, float* x,
                          void* stream);

/* Final RMSNorm of x_last (device fp32 [d]), logits = W_lm h (fp32 [vocab]),
 * first token = argmax, lowest index on ties.  ws: qcf_lm_head_workspace_size(). */
size_t qcf_lm_head_workspace_size(const qcf_dims* dims);
qcf_status qcf_lm_head(const qcf_model* m, const float* x_last, float* logits, int32_t* token, void* ws,
                       size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QCF_H_ */
