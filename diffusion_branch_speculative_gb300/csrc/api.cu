// C ABI of the folded multi-branch verification layer: argument checks,
// workspace layout, TMA descriptor encoding and the stage-by-stage launch
// sequence of specfold_layer_forward.  Everything is asynchronous on the
// caller's stream; nothing here allocates device memory.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <utility>

#include "sf_device.cuh"
#include "sf_internal.h"

namespace sf {

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) return 1;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (!v) {
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    v = v > 0 ? v : 1;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

int smem_limit_once(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPECFOLD_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, kernel})) return SPECFOLD_OK;
  // the kernel's static shared memory and the dynamic size together must fit
  // the per-block limit: a shape past it is unsupported, not a launch error
  cudaFuncAttributes fa;
  int optin = 0;
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return SPECFOLD_ECUDA;
  if (static_cast<long long>(fa.sharedSizeBytes) + bytes > optin) return SPECFOLD_EUNSUPPORTED;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return SPECFOLD_ECUDA;
  done.insert({dev, kernel});
  return SPECFOLD_OK;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("SPECFOLD_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

// Reads and clears the launch error state, so a rejected launch is reported
// by the call that made it and not again by every later one.
int check_launch() { return cudaGetLastError() == cudaSuccess ? SPECFOLD_OK : SPECFOLD_ECUDA; }

// ------------------------------------------------------------ TMA maps --
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

int make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t row_stride_elems,
                uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return SPECFOLD_ECUDA;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride_elems * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SPECFOLD_OK : SPECFOLD_ECUDA;
}

int make_map_3d(CUtensorMap* map, const void* base, uint64_t dim, uint64_t heads, uint64_t tokens,
                uint64_t head_stride, uint64_t token_stride, uint32_t box_tokens) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return SPECFOLD_ECUDA;
  const cuuint64_t dims[3] = {dim, heads, tokens};
  const cuuint64_t strides[2] = {head_stride * 2, token_stride * 2};
  const cuuint32_t box[3] = {64, 1, box_tokens};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SPECFOLD_OK : SPECFOLD_ECUDA;
}

// ------------------------------------------------------------- checks --
#define SF_TRY(x)              \
  do {                         \
    const int _rc = (x);       \
    if (_rc) return _rc;       \
  } while (0)

static bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static int esize(int dtype) { return dtype == SPECFOLD_BF16 ? 2 : 4; }
static bool dtype_ok(int dtype) { return dtype == SPECFOLD_BF16 || dtype == SPECFOLD_F32; }

static int check_rows(int B, int L) {
  if (B < 1 || L < 1) return SPECFOLD_EINVAL;
  if (static_cast<long long>(B) * L > SPECFOLD_MAX_ROWS) return SPECFOLD_ECAPACITY;
  return SPECFOLD_OK;
}

static int check_dims(const specfold_dims* d) {
  if (!d) return SPECFOLD_EINVAL;
  if (!dtype_ok(d->dtype)) return SPECFOLD_EINVAL;
  if (d->d_model <= 0 || d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 || d->ffn_dim <= 0)
    return SPECFOLD_EINVAL;
  if (!(d->rms_eps >= 0.f) || std::isinf(d->rms_eps)) return SPECFOLD_EINVAL;
  if (!(d->rope_theta >= 0.f) || std::isinf(d->rope_theta)) return SPECFOLD_EINVAL;
  if (d->gate_ref != 0 && d->gate_ref != 1) return SPECFOLD_EINVAL;
  if ((d->attn_rematch != 0 && d->attn_rematch != 1) || (d->ffn_gate != 0 && d->ffn_gate != 1))
    return SPECFOLD_EINVAL;
  if (d->head_dim != 64 && d->head_dim != 128) return SPECFOLD_EUNSUPPORTED;
  if (d->n_q_heads % d->n_kv_heads) return SPECFOLD_EUNSUPPORTED;
  if (d->d_model % 256) return SPECFOLD_EUNSUPPORTED;
  if ((d->n_q_heads * d->head_dim) % 128 || (d->n_kv_heads * d->head_dim) % 128) return SPECFOLD_EUNSUPPORTED;
  if (d->ffn_dim % 128) return SPECFOLD_EUNSUPPORTED;
  return SPECFOLD_OK;
}

static int check_weights(const specfold_weights* w) {
  if (!w) return SPECFOLD_EINVAL;
  const void* ps[9] = {w->g1, w->w_q, w->w_k, w->w_v, w->w_o, w->g2, w->w_gate, w->w_up, w->w_down};
  for (const void* p : ps) {
    if (!p) return SPECFOLD_EINVAL;
    if (!a16(p)) return SPECFOLD_EALIGN;
  }
  return SPECFOLD_OK;
}

static int check_view(const specfold_kv_view& v, int P) {
  if (P == 0) return SPECFOLD_OK;
  if (!v.ptr) return SPECFOLD_EINVAL;
  if (!a16(v.ptr)) return SPECFOLD_EALIGN;
  if (v.token_stride <= 0 || v.head_stride <= 0) return SPECFOLD_EINVAL;
  if (v.token_stride % 8 || v.head_stride % 8) return SPECFOLD_EALIGN;
  if (v.block_table) {
    if (v.page_size <= 0 || v.num_pages <= 0) return SPECFOLD_EINVAL;
    if (v.page_size % 8) return SPECFOLD_EUNSUPPORTED;
  }
  return SPECFOLD_OK;
}

// K and V of one call are both contiguous or both paged over one table.
static int check_views(const specfold_kv_view& k, const specfold_kv_view& v, int P) {
  SF_TRY(check_view(k, P));
  SF_TRY(check_view(v, P));
  if (P > 0 && (k.block_table != v.block_table || (k.block_table && k.page_size != v.page_size)))
    return SPECFOLD_EINVAL;
  return SPECFOLD_OK;
}



// ------------------------------------------------------ workspace layout --
static size_t up256(size_t x) { return (x + 255) / 256 * 256; }

static void layout(const specfold_dims* d, int B, int L, specfold_ws_layout* o) {
  const size_t R = static_cast<size_t>(B) * L;
  const size_t e = esize(d->dtype);
  const size_t nq = static_cast<size_t>(d->n_q_heads) * d->head_dim;
  const size_t nkv = static_cast<size_t>(d->n_kv_heads) * d->head_dim;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += up256(bytes);
    return at;
  };
  memset(o, 0, sizeof(*o));
  o->status = take(4);
  o->n_packed = take(4);
  o->fold = take(R);
  o->rel = take(R * 4);
  o->src = take(R * 4);
  o->packed_idx = take(R * 4);
  o->slot_of_row = take(R * 4);
  o->dep_rng = take(R * 8);
  o->dep_rows = take(R * 4);
  o->sync = take(gate_pack_sync_bytes());
  o->x1 = take(R * d->d_model * e);
  o->q = take(R * nq * e);
  o->block_k = take(R * nkv * e);
  o->block_v = take(R * nkv * e);
  o->attn_o = take(R * nq * e);
  o->a = take(R * d->d_model * e);
  o->x2 = take(R * d->d_model * e);
  o->g = take(R * d->ffn_dim * e);
  if (d->attn_rematch || d->ffn_gate) {  // the variant sublayer path only
    o->q_all = take(R * nq * e);
    o->all_idx = take(R * 4);
    o->n_all = take(4);
    o->a_all = take(R * d->d_model * e);
    o->fold_ffn = take(R);
    o->rel_ffn = take(R * 4);
    o->src_ffn = take(R * 4);
    o->packed_ffn = take(R * 4);
    o->slot_ffn = take(R * 4);
    o->n_ffn = take(4);
    o->dep_rng_ffn = take(R * 8);
    o->dep_rows_ffn = take(R * 4);
  }
  o->gemm_scratch = take(gemm_partial_floats() * 4);
  o->attn_scratch = take(attn_partial_bytes(static_cast<int>(R), d->n_q_heads / d->n_kv_heads, d->n_kv_heads,
                                            d->head_dim));
  o->total = off;
}

struct Scratch {
  float* partial;
  size_t partial_len;
  uint32_t* fill_bar;  // grid-barrier word of the down projection's two-pass finish
};

static Scratch layer_scratch(void* ws, const specfold_dims* d, int B, int L, const specfold_ws_layout& lo) {
  Scratch s;
  (void)d;
  (void)B;
  (void)L;
  s.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + lo.gemm_scratch);
  s.partial_len = gemm_partial_floats();
  // a word of the gate/pack sync header that the gate/pack barrier leaves alone
  // (that barrier uses the first word, and both return their word to zero)
  s.fill_bar = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + lo.sync + 64);
  return s;
}

template <typename T>
static T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

static void fill_scratch(GemmCall& c, const Scratch& s, uint32_t* status) {
  c.partial = s.partial;
  c.partial_len = s.partial_len;
  c.status = status;
}

// Stage events: recorded as graph event nodes while the stream is being
// captured (a plain record would become a capture-internal dependency).
static void record_stage_event(void* ev, cudaStream_t st) {
  if (!ev) return;  // entries may be NULL: only the given boundaries are recorded
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), st, cudaEventRecordExternal);
  else
    cudaEventRecord(static_cast<cudaEvent_t>(ev), st);
}

// ---------------------------------------------------------- stage bodies --
// bf16: the tcgen05 engine; fp32: the CUDA-core fp32 path.
static int gemm_call(int dtype, const GemmCall& c, cudaStream_t st, const RowNorm* rn = nullptr) {
  return dtype == SPECFOLD_F32 ? launch_gemm_f32(c, st, rn) : launch_gemm(c, st, rn);
}

static int stage_qkv(const specfold_dims* d, const specfold_weights* w, const void* X1, const int32_t* packed_idx,
                     const int32_t* n_dev, int R, void* Q, void* bK, void* bV, const Scratch& s, uint32_t* status,
                     cudaStream_t st) {
  GemmCall c;
  memset(&c, 0, sizeof(c));
  c.epi = EPI_QKV;
  c.A = X1;
  c.Mcap = R;
  c.K = d->d_model;
  c.n_dev = n_dev;
  c.nb = 3;
  c.b[0] = w->w_q;
  c.b[1] = w->w_k;
  c.b[2] = w->w_v;
  c.b_rows[0] = d->n_q_heads * d->head_dim;
  c.b_rows[1] = c.b_rows[2] = d->n_kv_heads * d->head_dim;
  c.N = c.b_rows[0] + 2 * c.b_rows[1];
  c.Y = Q;
  c.Yk = bK;
  c.Yv = bV;
  c.row_idx = packed_idx;
  c.n_q = d->n_q_heads;
  c.n_kv = d->n_kv_heads;
  c.hd = d->head_dim;
  fill_scratch(c, s, status);
  return gemm_call(d->dtype, c, st);
}

static int stage_attention(const specfold_dims* d, const void* Q, specfold_kv_view pk, specfold_kv_view pv, int P,
                           const void* bK, const void* bV, const int32_t* src, const int32_t* packed_idx,
                           const int32_t* n_dev, int B, int L, void* O, uint32_t* status, void* part,
                           size_t part_bytes, cudaStream_t st, const specfold_weights* w_ffn = nullptr,
                           bool n_early = false) {
  AttnCall a;
  memset(&a, 0, sizeof(a));
  a.n_early = n_early;
  if (w_ffn && d->dtype == SPECFOLD_BF16) {  // CTAs without work prefetch the next GEMMs' weights
    a.wo = w_ffn->w_o;
    a.wo_rows = d->d_model;
    a.wo_cols = d->n_q_heads * d->head_dim;
    a.ffn_w[0] = w_ffn->w_gate;
    a.ffn_w[1] = w_ffn->w_up;
    a.ffn_F = d->ffn_dim;
    a.ffn_d = d->d_model;
  }
  a.Q = Q;
  a.pk = pk;
  a.pv = pv;
  a.P = P;
  a.blockK = bK;
  a.blockV = bV;
  a.src = src;
  a.packed_idx = packed_idx;
  a.n_dev = n_dev;
  a.B = B;
  a.L = L;
  a.n_q = d->n_q_heads;
  a.n_kv = d->n_kv_heads;
  a.hd = d->head_dim;
  a.O = O;
  a.status = status;
  a.part = part;
  a.part_bytes = part_bytes;
  return d->dtype == SPECFOLD_F32 ? launch_attention_f32(a, st) : launch_attention(a, st);
}

static int stage_out_proj(const specfold_dims* d, const specfold_weights* w, const void* O,
                          const int32_t* packed_idx, const int32_t* n_dev, const void* H_in, int R, void* A,
                          const Scratch& s, uint32_t* status, cudaStream_t st, void* X2_fused = nullptr,
                          bool n_early = false) {
  GemmCall c;
  memset(&c, 0, sizeof(c));
  c.n_early = n_early;
  c.epi = EPI_RESID_PACKED;
  c.A = O;
  c.Mcap = R;
  c.K = d->n_q_heads * d->head_dim;
  c.n_dev = n_dev;
  c.nb = 1;
  c.b[0] = w->w_o;
  c.b_rows[0] = d->d_model;
  c.N = d->d_model;
  c.Y = A;
  c.ldy = d->d_model;
  c.resid = H_in;
  c.ldr = d->d_model;
  c.row_idx = packed_idx;
  fill_scratch(c, s, status);
  if (X2_fused) {
    const RowNorm rn{w->g2, d->rms_eps, X2_fused};
    return gemm_call(d->dtype, c, st, &rn);
  }
  return gemm_call(d->dtype, c, st);
}

// dep_rng / dep_rows (the folded rows grouped by source row, from the pack
// step) move the fold-fill into the down projection's finish kernel; without
// them a separate fold-fill kernel walks fold / src.
static int stage_ffn(const specfold_dims* d, const specfold_weights* w, const void* A, const int32_t* packed_idx,
                     const int32_t* n_dev, const void* H_in, const int32_t* src, const uint8_t* fold, int R,
                     void* H_out, void* X2, void* G, const Scratch& s, uint32_t* status, cudaStream_t st,
                     void* const* ev, int ev0, bool x2_ready, const int32_t* dep_rng = nullptr,
                     const int32_t* dep_rows = nullptr, bool n_early = false) {
  auto mark = [&](int i) {
    if (ev) record_stage_event(ev[i], st);
  };
  uint32_t* fill_bar = s.fill_bar;
  if (!x2_ready)
    SF_TRY(launch_rmsnorm_rows(d->dtype, A, nullptr, n_dev, R, d->d_model, w->g2, d->rms_eps, X2, st));
  GemmCall c;
  memset(&c, 0, sizeof(c));
  c.n_early = n_early;
  c.epi = EPI_SWIGLU;
  c.A = X2;
  c.Mcap = R;
  c.K = d->d_model;
  c.n_dev = n_dev;
  c.nb = 2;
  c.b[0] = w->w_gate;
  c.b[1] = w->w_up;
  c.b_rows[0] = c.b_rows[1] = d->ffn_dim;
  c.N = d->ffn_dim;
  c.Y = G;
  c.ldy = d->ffn_dim;
  fill_scratch(c, s, status);
  SF_TRY(gemm_call(d->dtype, c, st));
  mark(ev0 + 1);
  memset(&c, 0, sizeof(c));
  c.n_early = n_early;
  c.epi = EPI_RESID_SCATTER;
  c.A = G;
  c.Mcap = R;
  c.K = d->ffn_dim;
  c.n_dev = n_dev;
  c.nb = 1;
  c.b[0] = w->w_down;
  c.b_rows[0] = d->d_model;
  c.N = d->d_model;
  c.Y = H_out;
  c.ldy = d->d_model;
  c.resid = A;
  c.ldr = d->d_model;
  c.row_idx = packed_idx;
  fill_scratch(c, s, status);
  if (dep_rng && d->dtype == SPECFOLD_BF16) {  // the fp32 path fills with the fold-fill kernel
    c.dep_rng = dep_rng;
    c.dep_rows = dep_rows;
    c.hin = H_in;
    if (fill_bar) {
      c.fill_src = src;
      c.fill_bar = fill_bar;
    }
  } else {
    dep_rng = nullptr;
  }
  SF_TRY(gemm_call(d->dtype, c, st));
  mark(ev0 + 2);
  if (!dep_rng) SF_TRY(launch_fold_fill(d->dtype, fold, src, H_in, H_out, R, d->d_model, st));
  mark(ev0 + 3);
  return SPECFOLD_OK;
}

// Host-side checks of one layer call (everything but the workspace size).
static int check_layer_call(const specfold_dims* dims, const specfold_weights* w, const void* H_in,
                            const int32_t* parent, int B, int L, specfold_kv_view prefK, specfold_kv_view prefV,
                            int P, float tau, const void* H_out, const void* ws) {
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  SF_TRY(check_weights(w));
  if (!H_in || !parent || !H_out || !ws || P < 0) return SPECFOLD_EINVAL;
  if (!(tau >= 0.f)) return SPECFOLD_EINVAL;
  SF_TRY(check_views(prefK, prefV, P));
  if (!a16(H_in) || !a16(H_out) || !a16(ws)) return SPECFOLD_EALIGN;
  return SPECFOLD_OK;
}

// A stack's workspace: one layer workspace, then the [B, L, d] state buffer.
static size_t stack_ws_bytes(const specfold_dims* d, int B, int L, const specfold_ws_layout& lo) {
  return lo.total + up256(static_cast<size_t>(B) * L * d->d_model * esize(d->dtype));
}

static int launch_layer_gate(const specfold_dims* dims, const void* X, const int32_t* parent, int B, int L,
                             float tau, uint8_t* fold, float* rel, uint8_t* fold_hist, cudaStream_t st) {
  if (dims->gate_ref == 1)
    return launch_gate_source(dims->dtype, X, parent, B, L, dims->d_model, tau, fold, rel, st, fold_hist);
  return launch_gate(dims->dtype, X, parent, B, L, dims->d_model, tau, fold, rel, st, fold_hist);
}

// The layer as two sublayers (dims->attn_rematch or dims->ffn_gate): the
// attention sublayer gives A for every row (a_all), then the FFN sublayer
// packs its own rows of a_all (its own gate, or the first gate's decisions)
// and fills the rest with their FFN source's output plus their own A
// difference.
static int enqueue_layer_sublayers(const specfold_dims* dims, const specfold_weights* w, const void* H_in,
                                   const int32_t* parent, int B, int L, specfold_kv_view prefK,
                                   specfold_kv_view prefV, int P, float tau, void* H_out, void* ws,
                                   const specfold_ws_layout& lo, void* const* stage_events, uint8_t* fold_hist,
                                   int32_t* n_hist, cudaStream_t st) {
  const int R = B * L;
  const Scratch s = layer_scratch(ws, dims, B, L, lo);
  uint32_t* status = at<uint32_t>(ws, lo.status);
  uint8_t* fold = at<uint8_t>(ws, lo.fold);
  int32_t* src = at<int32_t>(ws, lo.src);
  int32_t* pidx = at<int32_t>(ws, lo.packed_idx);
  int32_t* slot = at<int32_t>(ws, lo.slot_of_row);
  int32_t* n_dev = at<int32_t>(ws, lo.n_packed);
  void* a_all = at<void>(ws, lo.a_all);
  auto mark = [&](int i) {
    if (stage_events) record_stage_event(stage_events[i], st);
  };
  mark(0);
  SF_TRY(launch_layer_gate(dims, H_in, parent, B, L, tau, fold, at<float>(ws, lo.rel), fold_hist, st));
  mark(1);
  SF_TRY(launch_select_pack(dims->dtype, fold, parent, B, L, dims->d_model, H_in, w->g1, dims->rms_eps, src, pidx,
                            slot, n_dev, at<void>(ws, lo.x1), status, st, n_hist));
  mark(2);
  SF_TRY(stage_qkv(dims, w, at<void>(ws, lo.x1), pidx, n_dev, R, at<void>(ws, lo.q), at<void>(ws, lo.block_k),
                   at<void>(ws, lo.block_v), s, status, st));
  if (dims->rope_theta > 0.f)
    SF_TRY(launch_rope(dims->dtype, at<void>(ws, lo.q), at<void>(ws, lo.block_k), pidx, n_dev, R, L, P,
                       dims->n_q_heads, dims->n_kv_heads, dims->head_dim, dims->rope_theta, st));
  mark(3);
  if (dims->attn_rematch) {
    // every row's query is its source's; attention and W_o run on all rows
    int32_t* all_idx = at<int32_t>(ws, lo.all_idx);
    int32_t* n_all = at<int32_t>(ws, lo.n_all);
    SF_TRY(launch_gather_query(dims->dtype, at<void>(ws, lo.q), src, slot, R, dims->n_kv_heads,
                               dims->n_q_heads / dims->n_kv_heads * dims->head_dim, at<void>(ws, lo.q_all), all_idx,
                               n_all, st));
    SF_TRY(stage_attention(dims, at<void>(ws, lo.q_all), prefK, prefV, P, at<void>(ws, lo.block_k),
                           at<void>(ws, lo.block_v), src, all_idx, n_all, B, L, at<void>(ws, lo.attn_o), status,
                           at<void>(ws, lo.attn_scratch), lo.total - lo.attn_scratch, st));
    mark(4);
    SF_TRY(stage_out_proj(dims, w, at<void>(ws, lo.attn_o), all_idx, n_all, H_in, R, a_all, s, status, st));
  } else {
    SF_TRY(stage_attention(dims, at<void>(ws, lo.q), prefK, prefV, P, at<void>(ws, lo.block_k),
                           at<void>(ws, lo.block_v), src, pidx, n_dev, B, L, at<void>(ws, lo.attn_o), status,
                           at<void>(ws, lo.attn_scratch), lo.total - lo.attn_scratch, st));
    mark(4);
    SF_TRY(stage_out_proj(dims, w, at<void>(ws, lo.attn_o), pidx, n_dev, H_in, R, at<void>(ws, lo.a), s, status, st));
    SF_TRY(launch_unpack_fill(dims->dtype, at<void>(ws, lo.a), src, slot, H_in, a_all, R, dims->d_model, st));
  }
  // FFN sublayer
  uint8_t* fold_f = fold;
  if (dims->ffn_gate) {
    fold_f = at<uint8_t>(ws, lo.fold_ffn);
    SF_TRY(launch_layer_gate(dims, a_all, parent, B, L, tau, fold_f, at<float>(ws, lo.rel_ffn), nullptr, st));
  }
  int32_t* src_f = at<int32_t>(ws, lo.src_ffn);
  int32_t* pidx_f = at<int32_t>(ws, lo.packed_ffn);
  int32_t* n_f = at<int32_t>(ws, lo.n_ffn);
  SF_TRY(launch_select_pack(dims->dtype, fold_f, parent, B, L, dims->d_model, a_all, w->g2, dims->rms_eps, src_f,
                            pidx_f, at<int32_t>(ws, lo.slot_ffn), n_f, at<void>(ws, lo.x2), status, st, nullptr,
                            at<int32_t>(ws, lo.dep_rng_ffn), at<int32_t>(ws, lo.dep_rows_ffn), at<void>(ws, lo.a)));
  mark(5);
  return stage_ffn(dims, w, at<void>(ws, lo.a), pidx_f, n_f, a_all, src_f, fold_f, R, H_out, at<void>(ws, lo.x2),
                   at<void>(ws, lo.g), s, status, st, stage_events, 5, true, at<int32_t>(ws, lo.dep_rng_ffn),
                   at<int32_t>(ws, lo.dep_rows_ffn));
}

// S1..S10 of one layer on `st` (arguments already checked).  fold_hist and
// n_hist, when given, receive copies of the layer's decisions and n.
static int enqueue_layer(const specfold_dims* dims, const specfold_weights* w, const void* H_in,
                         const int32_t* parent, int B, int L, specfold_kv_view prefK, specfold_kv_view prefV, int P,
                         float tau, void* H_out, void* ws, const specfold_ws_layout& lo,
                         void* const* stage_events, uint8_t* fold_hist, int32_t* n_hist, cudaStream_t st) {
  if (dims->attn_rematch || dims->ffn_gate)
    return enqueue_layer_sublayers(dims, w, H_in, parent, B, L, prefK, prefV, P, tau, H_out, ws, lo, stage_events,
                                   fold_hist, n_hist, st);
  const int R = B * L;
  const Scratch s = layer_scratch(ws, dims, B, L, lo);
  uint32_t* status = at<uint32_t>(ws, lo.status);
  uint8_t* fold = at<uint8_t>(ws, lo.fold);
  int32_t* src = at<int32_t>(ws, lo.src);
  int32_t* pidx = at<int32_t>(ws, lo.packed_idx);
  int32_t* n_dev = at<int32_t>(ws, lo.n_packed);
  auto mark = [&](int i) {
    if (stage_events) record_stage_event(stage_events[i], st);
  };
  mark(0);
  // S1-S3 in one launch (parent gate); the two-kernel form where the fused
  // kernel does not take the shape, or for the variant gate
  int rc = SPECFOLD_EUNSUPPORTED;
  if (dims->gate_ref == 0)
    rc = launch_gate_pack(dims->dtype, H_in, parent, B, L, dims->d_model, tau, w->g1, dims->rms_eps, fold,
                          at<float>(ws, lo.rel), src, pidx, at<int32_t>(ws, lo.slot_of_row), n_dev,
                          at<void>(ws, lo.x1), nullptr, nullptr,  // no dependents lists: the down
                          at<void>(ws, lo.sync), status, st, fold_hist, n_hist);  // finish fills from src
  if (rc == SPECFOLD_OK) {
    mark(1);  // the fused launch is the "gate" stage; "select_pack" is empty
  } else {
    if (rc != SPECFOLD_EUNSUPPORTED) return rc;
    SF_TRY(launch_layer_gate(dims, H_in, parent, B, L, tau, fold, at<float>(ws, lo.rel), fold_hist, st));
    mark(1);
    SF_TRY(launch_select_pack(dims->dtype, fold, parent, B, L, dims->d_model, H_in, w->g1, dims->rms_eps, src, pidx,
                              at<int32_t>(ws, lo.slot_of_row), n_dev, at<void>(ws, lo.x1), status, st, n_hist,
                              at<int32_t>(ws, lo.dep_rng), at<int32_t>(ws, lo.dep_rows)));
  }
  mark(2);
  SF_TRY(stage_qkv(dims, w, at<void>(ws, lo.x1), pidx, n_dev, R, at<void>(ws, lo.q), at<void>(ws, lo.block_k),
                   at<void>(ws, lo.block_v), s, status, st));
  if (dims->rope_theta > 0.f)
    SF_TRY(launch_rope(dims->dtype, at<void>(ws, lo.q), at<void>(ws, lo.block_k), pidx, n_dev, R, L, P,
                       dims->n_q_heads, dims->n_kv_heads, dims->head_dim, dims->rope_theta, st));
  mark(3);
  // from here on n_dev and packed_idx were written at least two launches
  // back (the QKV GEMM sits between), by a kernel that completed before the
  // QKV GEMM's programmatic wait returned: later kernels read them early
  SF_TRY(stage_attention(dims, at<void>(ws, lo.q), prefK, prefV, P, at<void>(ws, lo.block_k),
                         at<void>(ws, lo.block_v), src, pidx, n_dev, B, L, at<void>(ws, lo.attn_o), status,
                         at<void>(ws, lo.attn_scratch), lo.total - lo.attn_scratch, st, w, true));
  mark(4);
  SF_TRY(stage_out_proj(dims, w, at<void>(ws, lo.attn_o), pidx, n_dev, H_in, R, at<void>(ws, lo.a), s, status, st,
                        at<void>(ws, lo.x2), true));
  mark(5);
  return stage_ffn(dims, w, at<void>(ws, lo.a), pidx, n_dev, H_in, src, fold, R, H_out, at<void>(ws, lo.x2),
                   at<void>(ws, lo.g), s, status, st, stage_events, 5, true, at<int32_t>(ws, lo.dep_rng),
                   at<int32_t>(ws, lo.dep_rows), true);
}

}  // namespace sf

using namespace sf;

// ======================================================================
extern "C" {

size_t specfold_workspace_size(const specfold_dims* dims, int B, int L) {
  if (check_dims(dims) || check_rows(B, L)) return 0;
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  return lo.total;
}

int specfold_workspace_layout(const specfold_dims* dims, int B, int L, specfold_ws_layout* out) {
  if (!out) return SPECFOLD_EINVAL;
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  layout(dims, B, L, out);
  return SPECFOLD_OK;
}

size_t specfold_linear_workspace_size(int M, int N) {
  if (M <= 0 || N <= 0) return 0;
  return 256 + gemm_partial_floats() * 4;
}

int specfold_gate(int dtype, const void* H, const int32_t* parent, int B, int L, int d, float tau,
                  uint8_t* fold, float* rel_opt, void* stream) {
  if (!dtype_ok(dtype) || !H || !parent || !fold) return SPECFOLD_EINVAL;
  SF_TRY(check_rows(B, L));
  if (d <= 0) return SPECFOLD_EINVAL;
  if (!(tau >= 0.f)) return SPECFOLD_EINVAL;  // rejects NaN too
  if (d % 256) return SPECFOLD_EUNSUPPORTED;
  if (!a16(H)) return SPECFOLD_EALIGN;
  return launch_gate(dtype, H, parent, B, L, d, tau, fold, rel_opt, static_cast<cudaStream_t>(stream));
}

int specfold_gate_source(int dtype, const void* H, const int32_t* parent, int B, int L, int d, float tau,
                         uint8_t* fold, float* rel_opt, void* stream) {
  if (!dtype_ok(dtype) || !H || !parent || !fold) return SPECFOLD_EINVAL;
  SF_TRY(check_rows(B, L));
  if (d <= 0) return SPECFOLD_EINVAL;
  if (!(tau >= 0.f)) return SPECFOLD_EINVAL;
  if (d % 256) return SPECFOLD_EUNSUPPORTED;
  if (!a16(H)) return SPECFOLD_EALIGN;
  return launch_gate_source(dtype, H, parent, B, L, d, tau, fold, rel_opt, static_cast<cudaStream_t>(stream));
}

int specfold_resolve(const uint8_t* fold, const int32_t* parent, int B, int L, int32_t* src, uint32_t* status_opt,
                     void* stream) {
  if (!fold || !parent || !src) return SPECFOLD_EINVAL;
  SF_TRY(check_rows(B, L));
  return launch_select_pack(SPECFOLD_BF16, fold, parent, B, L, 0, nullptr, nullptr, 0.f, src, nullptr, nullptr,
                            nullptr, nullptr, status_opt, static_cast<cudaStream_t>(stream));
}

int specfold_pack(int dtype, const uint8_t* fold, const void* H, const void* g1, float eps, int B, int L, int d,
                  int32_t* packed_idx, int32_t* slot_of_row, int32_t* n_dev, void* X1, void* stream) {
  if (!dtype_ok(dtype) || !fold || !H || !g1 || !packed_idx || !slot_of_row || !n_dev || !X1)
    return SPECFOLD_EINVAL;
  SF_TRY(check_rows(B, L));
  if (d <= 0 || !(eps >= 0.f)) return SPECFOLD_EINVAL;
  if (d % 256) return SPECFOLD_EUNSUPPORTED;
  if (!a16(H) || !a16(g1) || !a16(X1)) return SPECFOLD_EALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // pack alone: no parent walk -- a folded non-root row is not recomputed
  return launch_select_pack(dtype, fold, nullptr, B, L, d, H, g1, eps, nullptr, packed_idx, slot_of_row, n_dev, X1,
                            nullptr, st);
}

int specfold_gate_pack(const specfold_dims* dims, const void* g1, const void* H, const int32_t* parent, int B, int L,
                       float tau, void* ws, size_t ws_bytes, void* stream) {
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  if (!g1 || !H || !parent || !ws) return SPECFOLD_EINVAL;
  if (!(tau >= 0.f)) return SPECFOLD_EINVAL;
  if (!a16(H) || !a16(g1) || !a16(ws)) return SPECFOLD_EALIGN;
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  if (ws_bytes < lo.total) return SPECFOLD_ECAPACITY;
  return launch_gate_pack(dims->dtype, H, parent, B, L, dims->d_model, tau, g1, dims->rms_eps, at<uint8_t>(ws, lo.fold),
                          at<float>(ws, lo.rel), at<int32_t>(ws, lo.src), at<int32_t>(ws, lo.packed_idx),
                          at<int32_t>(ws, lo.slot_of_row), at<int32_t>(ws, lo.n_packed), at<void>(ws, lo.x1),
                          at<int32_t>(ws, lo.dep_rng), at<int32_t>(ws, lo.dep_rows), at<void>(ws, lo.sync),
                          at<uint32_t>(ws, lo.status), static_cast<cudaStream_t>(stream));
}

int specfold_qkv(const specfold_dims* dims, const specfold_weights* w, const void* X1, const int32_t* packed_idx,
                 const int32_t* n_dev, int B, int L, void* Q, void* blockK, void* blockV, void* ws, size_t ws_bytes,
                 void* stream) {
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  SF_TRY(check_weights(w));
  if (!X1 || !packed_idx || !n_dev || !Q || !blockK || !blockV || !ws) return SPECFOLD_EINVAL;
  if (!a16(X1) || !a16(Q) || !a16(blockK) || !a16(blockV) || !a16(ws)) return SPECFOLD_EALIGN;
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  if (ws_bytes < lo.total) return SPECFOLD_ECAPACITY;
  const Scratch s = layer_scratch(ws, dims, B, L, lo);
  return stage_qkv(dims, w, X1, packed_idx, n_dev, B * L, Q, blockK, blockV, s, at<uint32_t>(ws, lo.status),
                   static_cast<cudaStream_t>(stream));
}

int specfold_rope(const specfold_dims* dims, void* Q, void* blockK, const int32_t* packed_idx, const int32_t* n_dev,
                  int B, int L, int P, void* stream) {
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  if (!Q || !blockK || !packed_idx || !n_dev || P < 0) return SPECFOLD_EINVAL;
  if (!a16(Q) || !a16(blockK)) return SPECFOLD_EALIGN;
  if (dims->rope_theta == 0.f) return SPECFOLD_OK;
  return launch_rope(dims->dtype, Q, blockK, packed_idx, n_dev, B * L, L, P, dims->n_q_heads, dims->n_kv_heads,
                     dims->head_dim, dims->rope_theta, static_cast<cudaStream_t>(stream));
}

int specfold_attention(const specfold_dims* dims, const void* Q, specfold_kv_view prefK, specfold_kv_view prefV,
                       int P, const void* blockK, const void* blockV, const int32_t* src, const int32_t* packed_idx,
                       const int32_t* n_dev, int B, int L, void* O, void* ws, size_t ws_bytes, void* stream) {
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  if (P < 0 || !Q || !blockK || !blockV || !src || !packed_idx || !n_dev || !O || !ws) return SPECFOLD_EINVAL;
  SF_TRY(check_views(prefK, prefV, P));
  if (!a16(Q) || !a16(blockK) || !a16(blockV) || !a16(O)) return SPECFOLD_EALIGN;
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  if (ws_bytes < lo.total) return SPECFOLD_ECAPACITY;
  return stage_attention(dims, Q, prefK, prefV, P, blockK, blockV, src, packed_idx, n_dev, B, L, O,
                         at<uint32_t>(ws, lo.status), at<void>(ws, lo.attn_scratch), lo.total - lo.attn_scratch,
                         static_cast<cudaStream_t>(stream));
}

int specfold_out_proj(const specfold_dims* dims, const specfold_weights* w, const void* O, const int32_t* packed_idx,
                      const int32_t* n_dev, const void* H_in, int B, int L, void* A, void* ws, size_t ws_bytes,
                      void* stream) {
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  SF_TRY(check_weights(w));
  if (!O || !packed_idx || !n_dev || !H_in || !A || !ws) return SPECFOLD_EINVAL;
  if (!a16(O) || !a16(H_in) || !a16(A)) return SPECFOLD_EALIGN;
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  if (ws_bytes < lo.total) return SPECFOLD_ECAPACITY;
  const Scratch s = layer_scratch(ws, dims, B, L, lo);
  return stage_out_proj(dims, w, O, packed_idx, n_dev, H_in, B * L, A, s, at<uint32_t>(ws, lo.status),
                        static_cast<cudaStream_t>(stream));
}

int specfold_ffn(const specfold_dims* dims, const specfold_weights* w, const void* A, const int32_t* packed_idx,
                 const int32_t* n_dev, const void* H_in, const int32_t* src, const uint8_t* fold, int B, int L,
                 void* H_out, void* ws, size_t ws_bytes, void* stream) {
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  SF_TRY(check_weights(w));
  if (!A || !packed_idx || !n_dev || !H_in || !src || !fold || !H_out || !ws) return SPECFOLD_EINVAL;
  if (!a16(A) || !a16(H_in) || !a16(H_out) || !a16(ws)) return SPECFOLD_EALIGN;
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  if (ws_bytes < lo.total) return SPECFOLD_ECAPACITY;
  const Scratch s = layer_scratch(ws, dims, B, L, lo);
  return stage_ffn(dims, w, A, packed_idx, n_dev, H_in, src, fold, B * L, H_out, at<void>(ws, lo.x2),
                   at<void>(ws, lo.g), s, at<uint32_t>(ws, lo.status), static_cast<cudaStream_t>(stream), nullptr,
                   0, false);
}

int specfold_layer_forward(const specfold_dims* dims, const specfold_weights* w, const void* H_in,
                           const int32_t* parent, int B, int L, specfold_kv_view prefK, specfold_kv_view prefV, int P,
                           float tau, void* H_out, void* ws, size_t ws_bytes, void* const* stage_events,
                           void* stream) {
  SF_TRY(check_layer_call(dims, w, H_in, parent, B, L, prefK, prefV, P, tau, H_out, ws));
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  if (ws_bytes < lo.total) return SPECFOLD_ECAPACITY;
  return enqueue_layer(dims, w, H_in, parent, B, L, prefK, prefV, P, tau, H_out, ws, lo, stage_events, nullptr,
                       nullptr, static_cast<cudaStream_t>(stream));
}

size_t specfold_stack_workspace_size(const specfold_dims* dims, int B, int L) {
  if (check_dims(dims) || check_rows(B, L)) return 0;
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  return stack_ws_bytes(dims, B, L, lo);
}

int specfold_stack_forward(const specfold_dims* dims, int n_layers, const specfold_weights* w, const void* H_in,
                           const int32_t* parent, int B, int L, const specfold_kv_view* prefK,
                           const specfold_kv_view* prefV, int P, float tau, void* H_out,
                           const specfold_stack_trace* trace, void* ws, size_t ws_bytes, void* stream) {
  if (n_layers < 1 || !w || !prefK || !prefV) return SPECFOLD_EINVAL;
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  // every layer is checked before anything is launched
  for (int l = 0; l < n_layers; ++l)
    SF_TRY(check_layer_call(dims, &w[l], H_in, parent, B, L, prefK[l], prefV[l], P, tau, H_out, ws));
  if (H_out == H_in) return SPECFOLD_EINVAL;
  const specfold_stack_trace tr = trace ? *trace : specfold_stack_trace{nullptr, nullptr, nullptr};
  if (tr.hidden && !a16(tr.hidden)) return SPECFOLD_EALIGN;
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  if (ws_bytes < stack_ws_bytes(dims, B, L, lo)) return SPECFOLD_ECAPACITY;
  const size_t R = static_cast<size_t>(B) * L;
  const size_t state_bytes = R * dims->d_model * esize(dims->dtype);
  if (tr.hidden) {
    // the caller's record of the states must not overlap H_in or H_out
    const uintptr_t h0 = reinterpret_cast<uintptr_t>(tr.hidden);
    const uintptr_t h1 = h0 + state_bytes * static_cast<size_t>(n_layers - 1);
    for (const void* p : {H_in, static_cast<const void*>(H_out)}) {
      const uintptr_t p0 = reinterpret_cast<uintptr_t>(p), p1 = p0 + state_bytes;
      if (p0 < h1 && h0 < p1) return SPECFOLD_EINVAL;
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Layer outputs alternate between H_out and the workspace's state buffer so
  // that the last layer writes H_out and no layer writes the state it reads.
  uint8_t* spare = at<uint8_t>(ws, lo.total);
  const void* x = H_in;
  for (int l = 0; l < n_layers; ++l) {
    void* y;
    if (l == n_layers - 1)
      y = H_out;
    else if (tr.hidden)
      y = static_cast<uint8_t*>(tr.hidden) + state_bytes * static_cast<size_t>(l);
    else
      y = ((n_layers - 1 - l) & 1) ? static_cast<void*>(spare) : H_out;
    SF_TRY(enqueue_layer(dims, &w[l], x, parent, B, L, prefK[l], prefV[l], P, tau, y, ws, lo, nullptr,
                         tr.fold ? tr.fold + R * static_cast<size_t>(l) : nullptr,
                         tr.n_packed ? tr.n_packed + l : nullptr, st));
    x = y;
  }
  return SPECFOLD_OK;
}

int specfold_linear(int dtype, const void* X, const void* W, int M, int N, int K, void* Y, void* ws, size_t ws_bytes,
                    void* stream) {
  if (!dtype_ok(dtype)) return SPECFOLD_EINVAL;
  if (!X || !W || !Y || !ws || M <= 0 || N <= 0 || K <= 0) return SPECFOLD_EINVAL;
  if (dtype == SPECFOLD_F32 ? (K % 32 || N % 32) : (K % 64 || N % 128)) return SPECFOLD_EUNSUPPORTED;
  if (!a16(X) || !a16(W) || !a16(Y) || !a16(ws)) return SPECFOLD_EALIGN;
  if (ws_bytes < specfold_linear_workspace_size(M, N)) return SPECFOLD_ECAPACITY;
  GemmCall c;
  memset(&c, 0, sizeof(c));
  c.epi = EPI_STORE;
  c.A = X;
  c.Mcap = M;
  c.K = K;
  c.n_dev = nullptr;
  c.nb = 1;
  c.b[0] = W;
  c.b_rows[0] = N;
  c.N = N;
  c.Y = Y;
  c.ldy = N;
  c.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + 256);
  c.partial_len = gemm_partial_floats();
  c.status = static_cast<uint32_t*>(ws);
  return gemm_call(dtype, c, static_cast<cudaStream_t>(stream));
}

struct specfold_graph_s {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  uint64_t kernels;  // kernels per replay
};

}  // extern "C"

// Captures enqueue(stream, capturing) into a graph: one eager call first
// (kernel attributes are set and arguments checked outside the capture), then
// the same call under a thread-local capture on a private stream.
template <typename F>
static int capture_graph(F enqueue, specfold_graph* graph) {
  if (!graph) return SPECFOLD_EINVAL;
  *graph = nullptr;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return SPECFOLD_ECUDA;
  int rc = enqueue(s, false);
  if (rc == SPECFOLD_OK && cudaStreamSynchronize(s) != cudaSuccess) rc = SPECFOLD_ECUDA;
  if (rc != SPECFOLD_OK) {
    cudaStreamDestroy(s);
    return rc;
  }
  const uint64_t k0 = g_launches.load();
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(s);
    return SPECFOLD_ECUDA;
  }
  rc = enqueue(s, true);
  const cudaError_t ce = cudaStreamEndCapture(s, &g);
  const uint64_t kernels = g_launches.load() - k0;
  g_launches.fetch_sub(kernels);  // captured, not launched
  cudaStreamDestroy(s);
  if (rc != SPECFOLD_OK || ce != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    return rc != SPECFOLD_OK ? rc : SPECFOLD_ECUDA;
  }
  cudaGraphExec_t exec = nullptr;
  if (cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return SPECFOLD_ECUDA;
  }
  specfold_graph h = new (std::nothrow) specfold_graph_s{g, exec, kernels};
  if (!h) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(g);
    return SPECFOLD_ECAPACITY;
  }
  *graph = h;
  return SPECFOLD_OK;
}

extern "C" {

int specfold_layer_graph_create(const specfold_dims* dims, const specfold_weights* w, const void* H_in,
                                const int32_t* parent, int B, int L, specfold_kv_view prefK, specfold_kv_view prefV,
                                int P, float tau, void* H_out, void* ws, size_t ws_bytes, void* const* stage_events,
                                specfold_graph* graph) {
  return capture_graph(
      [&](cudaStream_t s, bool capturing) {
        return specfold_layer_forward(dims, w, H_in, parent, B, L, prefK, prefV, P, tau, H_out, ws, ws_bytes,
                                      capturing ? stage_events : nullptr, s);
      },
      graph);
}

int specfold_stack_graph_create(const specfold_dims* dims, int n_layers, const specfold_weights* w,
                                const void* H_in, const int32_t* parent, int B, int L,
                                const specfold_kv_view* prefK, const specfold_kv_view* prefV, int P, float tau,
                                void* H_out, const specfold_stack_trace* trace, void* ws, size_t ws_bytes,
                                specfold_graph* graph) {
  return capture_graph(
      [&](cudaStream_t s, bool) {
        return specfold_stack_forward(dims, n_layers, w, H_in, parent, B, L, prefK, prefV, P, tau, H_out, trace, ws,
                                      ws_bytes, s);
      },
      graph);
}

int specfold_graph_launch(specfold_graph graph, void* stream) {
  if (!graph) return SPECFOLD_EINVAL;
  if (cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) != cudaSuccess) return SPECFOLD_ECUDA;
  count_launch(static_cast<int>(graph->kernels));
  return SPECFOLD_OK;
}

int specfold_graph_destroy(specfold_graph graph) {
  if (!graph) return SPECFOLD_EINVAL;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
  return SPECFOLD_OK;
}

int specfold_get_status(void* ws, uint32_t* status_out, void* stream) {
  if (!ws) return SPECFOLD_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return SPECFOLD_ECUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SPECFOLD_ECUDA;
  if (status_out) *status_out = v;
  if (v) {
    if (cudaMemsetAsync(ws, 0, 4, st) != cudaSuccess) return SPECFOLD_ECUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SPECFOLD_ECUDA;
    return SPECFOLD_EDEVICE;
  }
  return SPECFOLD_OK;
}

int specfold_read_n_packed(const void* ws, int B, int L, const specfold_dims* dims, int32_t* n_out, void* stream) {
  if (!ws || !n_out) return SPECFOLD_EINVAL;
  SF_TRY(check_dims(dims));
  SF_TRY(check_rows(B, L));
  specfold_ws_layout lo;
  layout(dims, B, L, &lo);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(n_out, static_cast<const uint8_t*>(ws) + lo.n_packed, 4, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return SPECFOLD_ECUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? SPECFOLD_OK : SPECFOLD_ECUDA;
}

const char* specfold_status_string(int s) {
  switch (s) {
    case SPECFOLD_OK: return "ok";
    case SPECFOLD_EINVAL: return "invalid argument";
    case SPECFOLD_EALIGN: return "pointer or stride not 16-byte aligned";
    case SPECFOLD_ECAPACITY: return "capacity exceeded (workspace or rows)";
    case SPECFOLD_EUNSUPPORTED: return "shape not supported by the kernels";
    case SPECFOLD_ECUDA: return "CUDA runtime error";
    case SPECFOLD_EDEVICE: return "device reported an error (see status bits)";
    default: return "unknown status";
  }
}

uint64_t specfold_launch_count(void) { return g_launches.load(); }

int specfold_selftest_timeout(uint32_t* status, uint64_t wait_ns, void* stream) {
  if (!status) return SPECFOLD_EINVAL;
  if (wait_ns > 1000000000ull) wait_ns = 1000000000ull;
  return launch_timeout_probe(status, wait_ns, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
