// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "specfold.h"
#include "sf_device.cuh"

namespace sf {

// ---- launch bookkeeping ----
void count_launch(int n = 1);
int num_sms();                        // SMs of the current device (cached per device)
int check_launch();                   // SPECFOLD_OK or SPECFOLD_ECUDA after a launch
// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (device, kernel); safe to call from several host threads.
int smem_limit_once(const void* kernel, int bytes);
template <typename... KArgs>
inline int smem_limit_once(void (*kernel)(KArgs...), int bytes) {
  return smem_limit_once(reinterpret_cast<const void*>(kernel), bytes);
}

// ---- row-wise kernels (rowwise.cu) ----
// gate: fold/rel per row; dtype bf16 or f32.  fold_hist (optional) receives
// a second copy of the decisions.
int launch_gate(int dtype, const void* H, const int32_t* parent, int B, int L, int d, float tau,
                uint8_t* fold, float* rel, cudaStream_t st, uint8_t* fold_hist = nullptr);
// variant gate: compare with the computed source of the parent's row
// (level-by-level over the draft graph, one CTA per block position).
int launch_gate_source(int dtype, const void* H, const int32_t* parent, int B, int L, int d, float tau,
                       uint8_t* fold, float* rel, cudaStream_t st, uint8_t* fold_hist = nullptr);
// resolve + pack scan (+ RMSNorm1 gather of the packed rows when X1 is
// given); parent may be null (pack alone); any output may be null.  n_hist
// (optional) receives a second copy of the packed-row count; dep_rng [R][2] /
// dep_rows [R] (optional) receive the folded rows grouped by their source row
// (for a recomputed row s, dep_rows[dep_rng[2s] .. dep_rng[2s+1])).
int launch_select_pack(int dtype, const uint8_t* fold, const int32_t* parent, int B, int L, int d,
                       const void* H, const void* g1, float eps, int32_t* src, int32_t* packed_idx,
                       int32_t* slot, int32_t* n_dev, void* X1, uint32_t* status, cudaStream_t st,
                       int32_t* n_hist = nullptr, int32_t* dep_rng = nullptr, int32_t* dep_rows = nullptr,
                       void* Xraw = nullptr);  // Xraw [R, d]: the packed rows themselves (needs X1)
// S1 + S2 + S3 fused (parent gate, one launch): gate decisions and r, the
// sources, the packed list, n, RMSNorm1 of the packed rows and the folded
// rows grouped by source, with one bounded grid-wide barrier between the
// gate and the pack.  sync: gate_pack_sync_bytes() of zero-initialised
// workspace (it returns to its initial state after every complete call).
// Returns SPECFOLD_EUNSUPPORTED for rows too wide for it.
size_t gate_pack_sync_bytes();
int launch_gate_pack(int dtype, const void* H, const int32_t* parent, int B, int L, int d, float tau,
                     const void* g1, float eps, uint8_t* fold, float* rel, int32_t* src, int32_t* packed_idx,
                     int32_t* slot, int32_t* n_dev, void* X1, int32_t* dep_rng, int32_t* dep_rows, void* sync,
                     uint32_t* status, cudaStream_t st, uint8_t* fold_hist = nullptr, int32_t* n_hist = nullptr);
// Y[k] = rmsnorm(X[idx ? idx[k] : k]) * g for k < n (n from n_dev, or R when null).
int launch_rmsnorm_rows(int dtype, const void* X, const int32_t* idx, const int32_t* n_dev,
                        int R, int d, const void* g, float eps, void* Y, cudaStream_t st);
// H_out[r] = H_out[s] + H_in[r] - H_in[s] for folded rows r, s = src[r].
int launch_fold_fill(int dtype, const uint8_t* fold, const int32_t* src, const void* H_in,
                     void* H_out, int R, int d, cudaStream_t st);
int launch_timeout_probe(uint32_t* status, uint64_t wait_ns, cudaStream_t st);
// Variant sublayer path: queries of every row from its source's packed row
// (Q layout [n_kv][R*g][hd], ghd = g*hd), plus the all-rows list; and the
// attention sublayer output of every row from the packed rows with the
// folded rows' own input difference.
int launch_gather_query(int dtype, const void* Q, const int32_t* src, const int32_t* slot, int R, int n_kv, int ghd,
                        void* Qall, int32_t* all_idx, int32_t* n_all, cudaStream_t st);
int launch_unpack_fill(int dtype, const void* Ap, const int32_t* src, const int32_t* slot, const void* H, void* Aall,
                       int R, int d, cudaStream_t st);
// Rotary embedding of the packed rows' queries and block keys in place.
int launch_rope(int dtype, void* Q, void* Kb, const int32_t* packed_idx, const int32_t* n_dev, int R, int L, int P,
                int n_q, int n_kv, int hd, float theta, cudaStream_t st);

// ---- tcgen05 GEMM (gemm_tc.cu) ----
enum GemmEpi : int {
  EPI_STORE = 0,          // Y[k][c] = acc                      (plain, identity rows)
  EPI_QKV = 1,            // Q head-group layout, K/V rows at row_idx[k]
  EPI_RESID_PACKED = 2,   // Y[k][c] = acc + resid[row_idx[k]][c]
  EPI_SWIGLU = 3,         // Y[k][f] = silu(acc_gate) * acc_up
  EPI_RESID_SCATTER = 4,  // Y[row_idx[k]][c] = acc + resid[k][c]
};

struct GemmCall {
  int epi;
  const void* A;          // [Mcap, K] bf16 row-major
  int Mcap;               // rows of A (and of the row-indexed outputs)
  int K;
  const int32_t* n_dev;   // rows to compute (device); null -> Mcap
  // B operands: `nb` weights stacked along N; for SWIGLU, b[0] = gate, b[1] = up
  const void* b[3];
  int b_rows[3];
  int nb;
  int N;                  // total output columns (SWIGLU: F)
  // epilogue
  void* Y;
  long long ldy;
  const void* resid;
  long long ldr;
  const int32_t* row_idx;
  void* Yk;               // QKV: block K / V outputs
  void* Yv;
  int n_q, n_kv, hd;      // QKV head layout
  // scratch: fp32 split-K partial tiles
  float* partial;
  size_t partial_len;     // floats, >= gemm_partial_floats()
  uint32_t* status;
  // RESID_SCATTER only, optional: fold-fill of the dependents of each packed
  // row (with s = row_idx[k], the rows dep_rows[dep_rng[2s] .. dep_rng[2s+1])
  // take Y[s] + hin[r] - hin[s]), run by the split finish kernel
  const int32_t* dep_rng;
  const int32_t* dep_rows;
  const void* hin;
  // RESID_SCATTER, optional (with dep_rng): the provenance table src[r] and a
  // zeroed grid-barrier word; the finish then fills by folded row in a second
  // pass after a grid barrier
  const int32_t* fill_src;
  uint32_t* fill_bar;
  // n_dev (and row_idx) were written at least two launches back, by a kernel
  // that had completed before this launch could start: read them through L2
  // before the programmatic wait instead of after it
  bool n_early;
};
size_t gemm_partial_floats();
// Optional RMSNorm of the finished rows of an EPI_RESID_PACKED GEMM (the
// output projection): out[k] = Y[k] * gain / sqrt(mean(Y[k]^2) + eps).
struct RowNorm {
  const void* gain;
  float eps;
  void* out;
};
int launch_gemm(const GemmCall& c, cudaStream_t st, const RowNorm* rn = nullptr);
// The same call for fp32 operands (simt_f32.cu): CUDA-core FMA, fp32 throughout.
int launch_gemm_f32(const GemmCall& c, cudaStream_t st, const RowNorm* rn = nullptr);

// ---- tcgen05 attention (attn_tc.cu) ----
struct AttnCall {
  const void* Q;          // [n_kv, R*g, hd]
  specfold_kv_view pk, pv;
  int P;
  const void* blockK;     // [R, n_kv, hd]
  const void* blockV;
  const int32_t* src;
  const int32_t* packed_idx;
  const int32_t* n_dev;
  int B, L, n_q, n_kv, hd;
  void* O;                // [R, n_q*hd]
  uint32_t* status;
  void* part;             // split-KV partials (attn_partial_bytes)
  size_t part_bytes;
  // optional: the SwiGLU weights [F, d] (gate, up); CTAs without a unit pull
  // their leading k-blocks into L2 for the FFN GEMM
  const void* ffn_w[2];
  int ffn_F, ffn_d;
  const void* wo;        // output-projection weight [wo_rows, wo_cols], prefetched before the FFN's
  int wo_rows, wo_cols;
  bool n_early;          // as GemmCall::n_early
};
int attn_slot_cap(int R, int g, int n_kv);
size_t attn_partial_bytes(int R, int g, int n_kv, int hd);
int launch_attention(const AttnCall& c, cudaStream_t st);
int launch_attention_f32(const AttnCall& c, cudaStream_t st);  // fp32 Q/K/V/O (simt_f32.cu)

// ---- TMA descriptors (api.cu) ----
// 2-D bf16 map over a row-major [rows, cols] matrix with a {64, box_rows}
// box and 128-byte swizzle.
int make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                uint64_t row_stride_elems, uint32_t box_rows);
// 3-D bf16 map {dim, heads, tokens} with strides in elements and a
// {64, 1, box_tokens} box, 128-byte swizzle.
int make_map_3d(CUtensorMap* map, const void* base, uint64_t dim, uint64_t heads, uint64_t tokens,
                uint64_t head_stride, uint64_t token_stride, uint32_t box_tokens);

}  // namespace sf
