/*
 * specfold.h -- C ABI of the GB300 (sm_103a) folded multi-branch verification
 * layer (SpecFold).
 *
 * The layer is one bidirectional transformer layer (RMSNorm, GQA attention,
 * SwiGLU FFN) evaluated over B draft branches of one L-token block that share
 * a prefix KV cache.  Rows whose layer input barely differs from the parent
 * branch are folded: they reuse the computed source row's output plus their
 * own input difference.  All other rows are packed into one batch and
 * recomputed.  Sources: the SpecFold explainer (blog.ontle.kr/blog/358) --
 * "observation" paragraph with Fig. 2 (the gate metric), the "mechanism"
 * paragraph (gate, packed batch, shared prefix cache without copies) and the
 * implementation note (gate, provenance and attention kernels, GQA,
 * zero-copy strided view); and the iitog.ru summary "SpecFold ускоряет
 * диффузионные языковые модели до 1,99x", key facts (folded attention and
 * FFN that keep the residual hidden states).
 *
 * Conventions for every entry point:
 *   - Pointers are device pointers owned by the caller unless stated.  The
 *     library never allocates device memory; scratch comes from a caller
 *     workspace (specfold_workspace_size) that must be zero-filled once after
 *     allocation (cudaMemset) and is left reusable by every successful call.
 *   - Every call is asynchronous on `stream` (a cudaStream_t, 0 = legacy
 *     default stream) and returns a status: 0 on success, a negative
 *     SPECFOLD_E* code for an error detected on the host before anything was
 *     launched.  Errors detected on the device (a bounded wait that ran out,
 *     an invalid draft-graph parent, a count beyond capacity) set bits in
 *     the workspace's device status word; read them with specfold_get_status.
 *   - Rows are r = b*L + i for branch b (0 = root / main branch) and block
 *     position i.  R = B*L is the row capacity.  The number of packed rows n
 *     stays on the device (n_dev) and kernels are sized for n = R, so a call
 *     never synchronises with the host.
 *   - Element type: dims.dtype.  SPECFOLD_BF16 runs the contractions on the
 *     tcgen05 tensor cores (fp32 accumulation); SPECFOLD_F32 keeps fp32
 *     throughout (CUDA-core fp32 FMA for the projections and attention, the
 *     tiny fp32 configuration).  All activations, weights and the prefix view
 *     use that type.
 *   - Kernels are launched with programmatic dependent launch, so each may
 *     start before the previous kernel in the stream has ended.  Inputs that
 *     no kernel of the call writes (weights, gains, the draft graph, the
 *     prefix view) may then be read before a kernel waits for its
 *     predecessor.  Everything a call reads must be complete in stream order
 *     before the call.  A caller's kernel that runs just before a call and
 *     releases its dependents early (griddepcontrol.launch_dependents) must
 *     not write those inputs after doing so.  Ordinary kernels, copies and
 *     memsets are complete before the call's first kernel starts.
 *   - Matrices are row-major.  Weights use the [out, in] layout.
 *   - Alignment: every pointer is 16-byte aligned; the prefix view strides are
 *     multiples of 8 elements (SPECFOLD_EALIGN otherwise).
 */
#ifndef SPECFOLD_H
#define SPECFOLD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- host status codes ---- */
#define SPECFOLD_OK            0
#define SPECFOLD_EINVAL       -1   /* null pointer, negative size, tau < 0 or NaN, ... */
#define SPECFOLD_EALIGN       -2   /* pointer or stride not 16-byte aligned */
#define SPECFOLD_ECAPACITY    -3   /* workspace too small, or B*L above SPECFOLD_MAX_ROWS */
#define SPECFOLD_EUNSUPPORTED -4   /* shape outside the kernels' tiling (see each call) */
#define SPECFOLD_ECUDA        -5   /* a CUDA runtime call failed (launch, attribute, ...) */
#define SPECFOLD_EDEVICE      -6   /* specfold_get_status: the device status word is non-zero */

/* ---- device status bits (specfold_get_status) ---- */
#define SPECFOLD_DEV_TIMEOUT    1u  /* a bounded wait inside a kernel ran out; outputs invalid */
#define SPECFOLD_DEV_BAD_PARENT 2u  /* parent[b] outside [0, b) for b > 0, or parent[0] != -1 */
#define SPECFOLD_DEV_BAD_PAGE   4u  /* a paged prefix view's block table names a page outside the pool */
/* With SPECFOLD_DEV_TIMEOUT, bit (SPECFOLD_DEV_SITE_SHIFT + site) names the
 * wait that ran out (the other waits of that kernel then give up without a
 * bit of their own), for a report:
 *   attention  0 loader: Q buffer free       1 loader: K/V stage free
 *              2 softmax: S ready            3 softmax: P V before a rescale
 *              4 softmax: P V before the last P   5 softmax: last P V
 *              6 MMA: P ready                7 MMA: Q loaded
 *              8 MMA: K/V loaded             9 MMA: S buffer free
 *             10 MMA: accumulators free
 *   GEMM      11 producer: stage free       12 MMA: accumulator free
 *             13 MMA: stage loaded          14 epilogue: accumulator ready
 *   gate/pack 15 row copies                 16 gains copy
 *             17 grid barrier
 *   probe     18 specfold_timeout_probe's wait */
#define SPECFOLD_DEV_SITE_SHIFT 8

#define SPECFOLD_MAX_ROWS 16384     /* largest B*L */

typedef enum { SPECFOLD_BF16 = 0, SPECFOLD_F32 = 1 } specfold_dtype;

/* Layer shape.  Constraints (SPECFOLD_EUNSUPPORTED otherwise): head_dim is 64
 * or 128; n_q_heads % n_kv_heads == 0; d_model % 256 == 0;
 * (n_q_heads*head_dim) % 128 == 0; (n_kv_heads*head_dim) % 128 == 0;
 * ffn_dim % 128 == 0. */
typedef struct {
  int d_model;      /* hidden size d */
  int n_q_heads;    /* query heads */
  int n_kv_heads;   /* key/value heads (GQA group g = n_q_heads / n_kv_heads) */
  int head_dim;     /* hd */
  int ffn_dim;      /* SwiGLU inner width F */
  float rms_eps;    /* RMSNorm epsilon (>= 0) */
  int dtype;        /* specfold_dtype */
  float rope_theta; /* rotary embedding base; 0 = no positional rotation inside the layer */
  int gate_ref;     /* 0: the gate compares a child with its parent's input (specfold_gate);
                       1: with the input of the row its parent's output comes from
                       (specfold_gate_source) */
  int attn_rematch; /* 1: the implementation note's correction read literally: every folded
                       row runs attention again (its source's query over its own branch's
                       block keys/values and the prefix) and the output projection; only
                       its FFN sublayer stays folded.  0: folded rows skip the whole layer. */
  int ffn_gate;     /* 1: the FFN sublayer has a gate of its own on the attention sublayer's
                       output A (same rule, tau and reference as the first gate) with its own
                       sources and packed list.  0: one gate for the whole layer. */
} specfold_dims;

/* Layer weights (device, [out, in] row-major, dims.dtype). */
typedef struct {
  const void* g1;      /* [d]            RMSNorm before attention */
  const void* w_q;     /* [n_q*hd, d] */
  const void* w_k;     /* [n_kv*hd, d] */
  const void* w_v;     /* [n_kv*hd, d] */
  const void* w_o;     /* [d, n_q*hd] */
  const void* g2;      /* [d]            RMSNorm before the FFN */
  const void* w_gate;  /* [F, d] */
  const void* w_up;    /* [F, d] */
  const void* w_down;  /* [d, F] */
} specfold_weights;

/* Zero-copy view of the shared prefix K (or V).
 * Contiguous (block_table == NULL): element (token t, kv head h, dim j) is
 * ptr[t*token_stride + h*head_stride + j].  Any slice of a larger (e.g.
 * fused K/V) cache can be passed without a copy.
 * Paged (block_table != NULL): ptr is a pool of num_pages pages of page_size
 * tokens; prefix token t lives in pool token
 * block_table[t / page_size] * page_size + t % page_size, i.e. at
 * ptr[(that pool token)*token_stride + h*head_stride + j].  The table
 * (device int32, ceil(P / page_size) entries) is shared by K and V: both
 * views of a call must give the same table and page size.  page_size is a
 * multiple of 8; a page id outside [0, num_pages) reads as zeros and sets
 * SPECFOLD_DEV_BAD_PAGE.  Pool tokens past P are never used, whatever they
 * hold. */
typedef struct {
  const void* ptr;
  int64_t token_stride;   /* elements, multiple of 8 */
  int64_t head_stride;    /* elements, multiple of 8 */
  const int32_t* block_table;  /* NULL: contiguous view */
  int32_t page_size;      /* tokens per page (paged only) */
  int32_t num_pages;      /* pages in the pool (paged only) */
} specfold_kv_view;

/* Byte offsets of the intermediates inside a layer workspace (for
 * inspection; all relative to the workspace base). */
typedef struct {
  size_t status;       /* uint32 device status word */
  size_t n_packed;     /* int32 n */
  size_t fold;         /* uint8  [R] */
  size_t rel;          /* float  [R] */
  size_t src;          /* int32  [R] */
  size_t packed_idx;   /* int32  [R] (first n valid) */
  size_t slot_of_row;  /* int32  [R] (-1 for folded rows) */
  size_t dep_rng;      /* int32  [R][2] for a recomputed row s: {beg, end}, the folded rows */
  size_t dep_rows;     /* int32  [R]    dep_rows[beg .. end) whose source is s (written by
                          specfold_gate_pack and specfold_pack; the layer call's fused gate/pack
                          leaves both unwritten: its down-projection finish fills from src) */
  size_t sync;         /* grid-barrier words (bytes 0 and 64), then int32 per-CTA counts from byte 128
                          (library use; each word returns to zero after every complete call) */
  size_t x1;           /* [R, d]        RMSNorm1 of packed rows */
  size_t q;            /* [n_kv, R*g, hd]  queries, head-group major */
  size_t block_k;      /* [R, n_kv, hd]  keys of recomputed rows (row r) */
  size_t block_v;      /* [R, n_kv, hd] */
  size_t attn_o;       /* [R, n_q*hd]   attention output, packed rows */
  size_t a;            /* [R, d]        attention sublayer output, packed rows (variant
                                        path: the FFN's packed rows of a_all) */
  size_t x2;           /* [R, d]        RMSNorm2 of a */
  size_t g;            /* [R, F]        silu(x2 Wg) * (x2 Wu) */
  /* the variant sublayer path (dims.attn_rematch or dims.ffn_gate); with
   * both flags 0 these regions are not reserved and their offsets are 0: */
  size_t q_all;        /* [n_kv, R*g, hd]  queries of every row (row r: its source's) */
  size_t all_idx;      /* int32 [R]     0 .. R-1, the all-rows list */
  size_t n_all;        /* int32         R */
  size_t a_all;        /* [R, d]        attention sublayer output of every row, row order */
  size_t fold_ffn;     /* uint8 [R]     FFN-sublayer gate decisions */
  size_t rel_ffn;      /* float [R] */
  size_t src_ffn;      /* int32 [R]     FFN sources */
  size_t packed_ffn;   /* int32 [R]     FFN packed list (first n_ffn valid) */
  size_t slot_ffn;     /* int32 [R] */
  size_t n_ffn;        /* int32 */
  size_t dep_rng_ffn;  /* int32 [R][2] */
  size_t dep_rows_ffn; /* int32 [R] */
  size_t gemm_scratch; /* fp32 split-K partial sums */
  size_t attn_scratch; /* fp32 split-KV attention partials */
  size_t total;        /* total bytes */
} specfold_ws_layout;

/* Number of stage events specfold_layer_forward records when given them:
 * before the gate, after the gate, after resolve + pack + RMSNorm1, after the
 * QKV projection, after attention, after the output projection (+ RMSNorm2),
 * after the SwiGLU GEMM, after the down projection, after the fold-fill. */
#define SPECFOLD_STAGE_EVENTS 9

/* ------------------------------------------------------------------ */
/* S1 gate.  Explainer, Fig. 2 paragraph: r(b,i) = |H_b[i] - H_p[i]| / |H_p[i]|
 * on the layer input, p = parent[b] (the first parent of a multi-parent
 * node).  fold[r] = 1 iff sum(delta^2) < tau^2 * sum(H_p^2), or the row equals
 * its parent row and tau > 0 (so tau = 0 folds nothing).  Root rows: fold 0,
 * rel -1.  A parent outside [0, b) makes the row recompute (fold 0).
 *   H       [B, L, d] dims-dtype          parent  int32 [B]
 *   fold    uint8 [B*L] (out)             rel_opt float [B*L] (out, may be NULL)
 * d % 256 == 0. */
int specfold_gate(int dtype, const void* H, const int32_t* parent, int B, int L, int d,
                  float tau, uint8_t* fold, float* rel_opt, void* stream);

/* S1 variant: the gate against the computed source.  As specfold_gate, but
 * child row (b, i) is compared with row (s, i), s the branch whose row the
 * parent's output at position i comes from (the parent itself if it was
 * recomputed, else the parent's source): r = |H_b[i] - H_s[i]| / |H_s[i]|.
 * A chain of folds then never reuses an output whose input is more than
 * tau away.  Decisions follow the draft graph level by level (one CTA per
 * position i).  Same arguments and outputs as specfold_gate. */
int specfold_gate_source(int dtype, const void* H, const int32_t* parent, int B, int L, int d,
                         float tau, uint8_t* fold, float* rel_opt, void* stream);

/* S2 resolve.  Explainer, implementation note (provenance kernel): src[r] = r
 * for a recomputed row, else src of the same position in the parent branch,
 * following the fold chain to the row actually computed.  A bad parent
 * (outside [0, b)) ends the chain at that row and sets SPECFOLD_DEV_BAD_PARENT
 * in *status_opt (device uint32, may be NULL).
 *   fold uint8 [B*L], parent int32 [B] -> src int32 [B*L] */
int specfold_resolve(const uint8_t* fold, const int32_t* parent, int B, int L,
                     int32_t* src, uint32_t* status_opt, void* stream);

/* S3 pack.  Explainer, "mechanism" paragraph and implementation note: every
 * recomputed row of every branch goes into one packed batch, branch-major and
 * position-ascending (increasing r), and is RMS-normalised:
 *   X1[k] = H[packed_idx[k]] * g1 / sqrt(mean(H^2) + eps)
 *   fold uint8 [B*L], H [B, L, d], g1 [d]
 *   -> packed_idx int32 [B*L] (first n valid), slot_of_row int32 [B*L]
 *      (-1 for folded rows), n_dev int32 [1], X1 [B*L, d] (first n rows). */
int specfold_pack(int dtype, const uint8_t* fold, const void* H, const void* g1, float eps,
                  int B, int L, int d, int32_t* packed_idx, int32_t* slot_of_row,
                  int32_t* n_dev, void* X1, void* stream);

/* S1 + S2 + S3 in one launch (the parent gate), as specfold_layer_forward
 * runs them: the gate decisions and r, the sources, the packed list, n,
 * RMSNorm1 of the packed rows and the folded rows grouped by source, all
 * written into the layer workspace ws (offsets: specfold_workspace_layout;
 * fields fold, rel, src, packed_idx, slot_of_row, n_packed, x1, dep_rng,
 * dep_rows).  Same rules as the three calls above (explainer, "observation"
 * and "mechanism" paragraphs, implementation note).  One CTA per SM at most,
 * meeting once at a bounded grid barrier: if that wait runs out (another
 * kernel holding SMs for over a second) the call sets SPECFOLD_DEV_TIMEOUT and
 * the workspace must be zeroed again before its next use.  dims gives d, eps
 * and the dtype; rows wider than 4096 bf16 (2048 fp32) elements, or draft
 * graphs too large for the shared memory of one CTA, give
 * SPECFOLD_EUNSUPPORTED (use the three calls above). */
int specfold_gate_pack(const specfold_dims* dims, const void* g1, const void* H, const int32_t* parent, int B,
                       int L, float tau, void* ws, size_t ws_bytes, void* stream);

/* S4 QKV projection of the packed rows (one transformer layer's attention
 * input projections).  Q goes to the head-group-major layout
 * Q[h_kv][k*g + j][hd] (query head h_kv*g + j of packed row k, R*g rows per
 * KV head); keys/values of packed row k go to row packed_idx[k] of
 * blockK/blockV [B*L, n_kv, hd].  Rows of folded positions are not written.
 * ws: a layer workspace (split-K scratch, status). */
int specfold_qkv(const specfold_dims* dims, const specfold_weights* w, const void* X1,
                 const int32_t* packed_idx, const int32_t* n_dev, int B, int L,
                 void* Q, void* blockK, void* blockV, void* ws, size_t ws_bytes, void* stream);

/* S4b rotary position embedding (rotate-half convention of the Qwen/Llama
 * families; the pages put no positional encoding inside the layer, so this
 * is the real-model follow-on).  Only when dims->rope_theta > 0: the queries
 * of every packed row k < n and the block keys of its row r = packed_idx[k]
 * are rotated in place, block position i = r % L sitting at absolute
 * position P + i: for j < hd/2 the pair (x[j], x[j + hd/2]) turns by the
 * angle (P + i) * rope_theta^(-2j/hd).  The prefix keys are taken as already
 * rotated (a KV cache stores them so); values are never rotated.  Q and
 * blockK use the layouts of specfold_qkv.  Returns SPECFOLD_OK without
 * launching anything when rope_theta == 0. */
int specfold_rope(const specfold_dims* dims, void* Q, void* blockK, const int32_t* packed_idx,
                  const int32_t* n_dev, int B, int L, int P, void* stream);

/* S5 folded attention.  Explainer, implementation note: FlashAttention-style
 * streaming with GQA; the shared prefix K/V is read through the strided view
 * (never copied per branch); packed row k of branch b attends to all P prefix
 * keys and to the L block keys of its own branch, block key j being row
 * src[b*L + j] of blockK/blockV (a folded position uses its resolved source's
 * key/value).  No mask inside the block, no attention across branches,
 * softmax scale 1/sqrt(hd).
 *   Q as written by specfold_qkv -> O [B*L, n_q*hd] (packed rows, first n). */
int specfold_attention(const specfold_dims* dims, const void* Q, specfold_kv_view prefK,
                       specfold_kv_view prefV, int P, const void* blockK, const void* blockV,
                       const int32_t* src, const int32_t* packed_idx, const int32_t* n_dev,
                       int B, int L, void* O, void* ws, size_t ws_bytes, void* stream);

/* S6 output projection + residual: A[k] = H[packed_idx[k]] + O[k] w_o^T. */
int specfold_out_proj(const specfold_dims* dims, const specfold_weights* w, const void* O,
                      const int32_t* packed_idx, const int32_t* n_dev, const void* H_in,
                      int B, int L, void* A, void* ws, size_t ws_bytes, void* stream);

/* S7-S10 folded FFN.  iitog.ru summary (key facts) and explainer
 * ("keep own difference"): for packed rows
 *   X2 = rmsnorm(A) * g2;  G = silu(X2 Wg^T) * (X2 Wu^T);
 *   H_out[packed_idx[k]] = A[k] + G[k] Wd^T
 * then for every folded row r with s = src[r]:
 *   H_out[r] = H_out[s] + (H_in[r] - H_in[s]).
 * X2 and G live in the workspace. */
int specfold_ffn(const specfold_dims* dims, const specfold_weights* w, const void* A,
                 const int32_t* packed_idx, const int32_t* n_dev, const void* H_in,
                 const int32_t* src, const uint8_t* fold, int B, int L, void* H_out,
                 void* ws, size_t ws_bytes, void* stream);

/* S1-S10: the whole folded layer.  H_in [B, L, d], parent int32 [B] (first
 * parents, parent[0] = -1, parent[b] < b), prefix views of P tokens, tau >= 0
 * (0 = folding off: the dense multi-branch verify through the same kernels).
 * Writes H_out [B, L, d]; intermediates stay in ws (specfold_workspace_layout).
 * With dims.attn_rematch or dims.ffn_gate the layer runs as two sublayers:
 *   attention: gate, pack and QKV as above; with attn_rematch, attention and
 *     the output projection run on every row (row r's query is its source's),
 *     giving A for all rows; without it, on the packed rows, and a folded row
 *     takes A[r] = A[s] + (H_in[r] - H_in[s]);
 *   FFN: with ffn_gate a second gate on A (fold_ffn, src_ffn, packed_ffn);
 *     without it the first gate's decisions; the FFN runs on its packed rows
 *     and a folded row r with FFN source s takes
 *     H_out[r] = H_out[s] + (A[r] - A[s]).
 * With both 0 this is the layer above: H_out[r] = H_out[s] + (H_in[r] - H_in[s]).
 * stage_events: NULL, or SPECFOLD_STAGE_EVENTS cudaEvent_t handles recorded
 * on `stream` at the stage boundaries listed at SPECFOLD_STAGE_EVENTS; a NULL
 * entry skips that boundary. */
int specfold_layer_forward(const specfold_dims* dims, const specfold_weights* w,
                           const void* H_in, const int32_t* parent, int B, int L,
                           specfold_kv_view prefK, specfold_kv_view prefV, int P, float tau,
                           void* H_out, void* ws, size_t ws_bytes,
                           void* const* stage_events, void* stream);

/* CUDA graph of one specfold_layer_forward call.  The library captures the
 * whole launch sequence once (on a private stream, thread-local capture) and
 * replays it with a single graph launch, which removes the per-kernel host
 * launch cost.  Every pointer, the shape, tau and the optional stage events
 * are fixed at creation: to run on new inputs, write them into the same H_in
 * / parent buffers before each launch.  Returns SPECFOLD_OK and sets *graph,
 * or an error code (nothing is captured then). */
typedef struct specfold_graph_s* specfold_graph;
int specfold_layer_graph_create(const specfold_dims* dims, const specfold_weights* w,
                                const void* H_in, const int32_t* parent, int B, int L,
                                specfold_kv_view prefK, specfold_kv_view prefV, int P, float tau,
                                void* H_out, void* ws, size_t ws_bytes,
                                void* const* stage_events, specfold_graph* graph);
/* ---- stack of layers ---------------------------------------------- */
/* Optional per-layer records of a stack call (all device pointers, each may
 * be NULL):
 *   hidden    [n_layers - 1, B, L, d] dims.dtype: the input of layers
 *             1 .. n_layers-1 (= the output of layers 0 .. n_layers-2).
 *             When NULL those states live in the workspace and are
 *             overwritten as the stack proceeds.
 *   fold      uint8 [n_layers, B*L]: each layer's gate decisions.
 *   n_packed  int32 [n_layers]: each layer's packed-row count n (the
 *             recompute fraction of layer l is n_packed[l] / (B*L)).
 * With dims.attn_rematch or dims.ffn_gate set, fold and n_packed record the
 * layer's first gate only: attention and the output projection then run on
 * every row (attn_rematch), and the FFN sublayer's own decisions and packed
 * count (ffn_gate) are not recorded. */
typedef struct specfold_stack_trace {
  void* hidden;
  uint8_t* fold;
  int32_t* n_packed;
} specfold_stack_trace;

/* Workspace bytes for a stack of layers of this shape: a layer workspace
 * plus one [B, L, d] buffer for the states between layers.  0 if invalid. */
size_t specfold_stack_workspace_size(const specfold_dims* dims, int B, int L);

/* A stack of n_layers folded layers: layer l reads layer l-1's output
 * (layer 0 reads H_in) and the last layer writes H_out.  Explainer,
 * "mechanism" paragraph (automatic release of a fold) and appendix D (how
 * the recompute fraction changes with depth): the gate runs again at every
 * layer on that layer's own input, so a row folded at layer l is recomputed
 * at layer l+1 when its difference to the parent's new input reaches tau.
 * w, prefK and prefV are HOST arrays of n_layers entries (each layer's own
 * weights and prefix view; the pointers inside are device pointers).  Same
 * shape for every layer, same parent table and tau.  trace may be NULL.
 * ws: specfold_stack_workspace_size bytes.  H_out must not alias H_in or
 * trace->hidden.  Errors as for specfold_layer_forward; an invalid layer
 * makes the call return before anything is launched. */
int specfold_stack_forward(const specfold_dims* dims, int n_layers, const specfold_weights* w,
                           const void* H_in, const int32_t* parent, int B, int L,
                           const specfold_kv_view* prefK, const specfold_kv_view* prefV, int P,
                           float tau, void* H_out, const specfold_stack_trace* trace,
                           void* ws, size_t ws_bytes, void* stream);

/* CUDA graph of one specfold_stack_forward call (same rules as
 * specfold_layer_graph_create; the host arrays are read at creation only). */
int specfold_stack_graph_create(const specfold_dims* dims, int n_layers, const specfold_weights* w,
                                const void* H_in, const int32_t* parent, int B, int L,
                                const specfold_kv_view* prefK, const specfold_kv_view* prefV, int P,
                                float tau, void* H_out, const specfold_stack_trace* trace,
                                void* ws, size_t ws_bytes, specfold_graph* graph);

/* Enqueue one replay on `stream`. */
int specfold_graph_launch(specfold_graph graph, void* stream);
/* Release the graph (after its launches have completed). */
int specfold_graph_destroy(specfold_graph graph);

/* Plain packed GEMM through the same tcgen05 engine: Y[M, N] = X[M, K] W^T
 * with W [N, K]; Y in dims-dtype.  K % 64 == 0, N % 128 == 0. */
int specfold_linear(int dtype, const void* X, const void* W, int M, int N, int K, void* Y,
                    void* ws, size_t ws_bytes, void* stream);

/* The plain GEMM of specfold_linear for callers that cannot allocate device
 * memory: a plain C caller that holds only its inputs and outputs and has no
 * device allocator of its own, or a serving runtime that owns all device
 * memory and forbids allocation after warm-up.  The SpecFold pages have no
 * counterpart; this is a library convenience.
 * Y[M, N] = X[M, K] W^T, the same product as specfold_linear but with its own
 * split-K schedule (a grid capped at 128 CTAs), so the two can differ in the
 * last bits of a sum.  No workspace argument: the split-K scratch is a
 * 16 MiB static device array inside the library, held by every GPU that
 * loads it until the process exits.  Limits: M <= SPECFOLD_MAX_ROWS (larger
 * M: SPECFOLD_ECAPACITY); K % 64 == 0 and N % 128 == 0
 * (SPECFOLD_EUNSUPPORTED); at most 128 CTAs, so it can be slower than
 * specfold_linear on large problems.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  Every call shares the one
 * array: calls that overlap on the GPU (other streams, or other host threads)
 * race and must be serialised by the caller.  The scratch is fully rewritten
 * before it is read, so a call needs nothing cleared from the previous one.
 * A bounded wait that runs out cannot be reported (there is no status word). */
int specfold_linear_noalloc(int dtype, const void* X, const void* W, int M, int N, int K, void* Y,
                            void* stream);

/* Workspace bytes for a layer of this shape and B*L rows (host only, no GPU
 * needed).  0 if the shape is invalid. */
size_t specfold_workspace_size(const specfold_dims* dims, int B, int L);

/* Workspace bytes for specfold_linear with M rows and N columns. */
size_t specfold_linear_workspace_size(int M, int N);

/* Offsets of the intermediates for this shape.  Returns SPECFOLD_OK or
 * SPECFOLD_EINVAL / SPECFOLD_EUNSUPPORTED. */
int specfold_workspace_layout(const specfold_dims* dims, int B, int L, specfold_ws_layout* out);

/* Synchronises `stream`, copies the workspace's device status word to
 * *status_out (may be NULL) and clears it.  Returns SPECFOLD_OK if it was 0,
 * SPECFOLD_EDEVICE if not, SPECFOLD_ECUDA if the copy failed. */
int specfold_get_status(void* ws, uint32_t* status_out, void* stream);

/* Reads the packed-row count n of the last layer call on `stream`
 * (synchronises the stream). */
int specfold_read_n_packed(const void* ws, int B, int L, const specfold_dims* dims,
                           int32_t* n_out, void* stream);

/* Static string for a status code. */
const char* specfold_status_string(int status);

/* Kernels this library has launched in this process (host counter). */
uint64_t specfold_launch_count(void);

/* Self-test of the bounded-wait path: launches one block that waits on an
 * mbarrier nobody arrives at, for at most wait_ns nanoseconds (capped at
 * 1e9); the wait runs out, the kernel sets SPECFOLD_DEV_TIMEOUT in *status
 * (device uint32) and returns.  The GPU context stays usable. */
int specfold_selftest_timeout(uint32_t* status, uint64_t wait_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SPECFOLD_H */
