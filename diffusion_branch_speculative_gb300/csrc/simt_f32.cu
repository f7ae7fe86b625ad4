// fp32 path of the layer (the tiny fp32 configuration): the projections and
// the folded attention in plain fp32 FMA on the CUDA cores, so results keep
// fp32 precision (the tensor cores' tf32 would drop to a 10-bit mantissa).
// The row-wise kernels (gate, pack, RMSNorm, fold-fill) are shared with the
// bf16 path; only the two contractions differ.  Sizes here are small: the
// kernels favour plainness over speed.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "sf_device.cuh"
#include "sf_internal.h"

namespace sf {
namespace {

constexpr int kT = 32;  // output tile (rows x columns) and K step

struct GemmF32 {
  const float* A;
  int Mcap, K, N;
  const int32_t* n_dev;
  const float* b[3];
  int col0[3];
  int nb;
  int epi;
  float* Y;
  long long ldy;
  const float* resid;
  long long ldr;
  const int32_t* row_idx;
  float* Yk;
  float* Yv;
  int n_q, n_kv, hd, g, R;
};

__device__ __forceinline__ const float* weight_row(const GemmF32& p, int c) {
  int j = 0;
  while (j + 1 < p.nb && c >= p.col0[j + 1]) ++j;
  return p.b[j] + static_cast<size_t>(c - p.col0[j]) * p.K;
}

// C[k][c] = sum_j A[k][j] W[c][j] over a 32 x 32 tile, K in steps of 32;
// thread (tx, ty) owns column tx of rows ty, ty + 8, ty + 16, ty + 24.
// SwiGLU (epi 3): c is a feature; b[0] holds the gate rows, b[1] the up rows.
__global__ void __launch_bounds__(256) gemm_f32_kernel(const GemmF32 p) {
  __shared__ float sA[kT][kT + 1];
  __shared__ float sB[kT][kT + 1];
  __shared__ float sU[kT][kT + 1];
  pdl_wait();
  pdl_trigger();
  const int n = p.n_dev ? min(max(p.n_dev[0], 0), p.Mcap) : p.Mcap;
  const int m0 = blockIdx.y * kT, c0 = blockIdx.x * kT;
  if (m0 >= n) return;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const bool swiglu = p.epi == EPI_SWIGLU;
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < p.K; k0 += kT) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int rr = ty + 8 * q;
      sA[rr][tx] = m0 + rr < n ? p.A[static_cast<size_t>(m0 + rr) * p.K + k0 + tx] : 0.f;
      const int c = c0 + rr;
      if (swiglu) {
        sB[rr][tx] = p.b[0][static_cast<size_t>(c) * p.K + k0 + tx];
        sU[rr][tx] = p.b[1][static_cast<size_t>(c) * p.K + k0 + tx];
      } else {
        sB[rr][tx] = weight_row(p, c)[k0 + tx];
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kT; ++kk) {
      const float wb = sB[tx][kk];
      const float wu = swiglu ? sU[tx][kk] : 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = sA[ty + 8 * q][kk];
        acc[q] = fmaf(a, wb, acc[q]);
        if (swiglu) accu[q] = fmaf(a, wu, accu[q]);
      }
    }
    __syncthreads();
  }
  const int c = c0 + tx;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int k = m0 + ty + 8 * q;
    if (k >= n) continue;
    const float x = acc[q];
    switch (p.epi) {
      case EPI_STORE:
        p.Y[static_cast<size_t>(k) * p.ldy + c] = x;
        break;
      case EPI_RESID_PACKED:
        p.Y[static_cast<size_t>(k) * p.ldy + c] = x + p.resid[static_cast<size_t>(p.row_idx[k]) * p.ldr + c];
        break;
      case EPI_RESID_SCATTER:
        p.Y[static_cast<size_t>(p.row_idx[k]) * p.ldy + c] = x + p.resid[static_cast<size_t>(k) * p.ldr + c];
        break;
      case EPI_SWIGLU:
        p.Y[static_cast<size_t>(k) * p.ldy + c] = x / (1.f + expf(-x)) * accu[q];
        break;
      default: {  // EPI_QKV
        const int nq = p.n_q * p.hd, nkv = p.n_kv * p.hd;
        if (c < nq) {
          const int head = c / p.hd, j = c - head * p.hd;
          const int hk = head / p.g, hg = head - hk * p.g;
          p.Y[((static_cast<size_t>(hk) * p.R + k) * p.g + hg) * p.hd + j] = x;
        } else {
          const bool is_k = c < nq + nkv;
          const int cc = is_k ? c - nq : c - nq - nkv;
          (is_k ? p.Yk : p.Yv)[static_cast<size_t>(p.row_idx[k]) * nkv + cc] = x;
        }
      }
    }
  }
}

struct AttnF32 {
  const float* Q;       // [n_kv][R*g][hd]
  const float* pk;      // prefix K / V base (contiguous view or page pool)
  const float* pv;
  long long k_ts, k_hs, v_ts, v_hs;
  const int32_t* table; // paged prefix (null: contiguous)
  int page_size, num_pages;
  const float* bK;      // [R][n_kv][hd]
  const float* bV;
  const int32_t* src;
  const int32_t* packed_idx;
  const int32_t* n_dev;
  float* O;             // [R][n_q*hd]
  int P, L, R, n_q, n_kv, g, hd;
  uint32_t* status;
};

// One warp per (packed row k, query head h): online softmax over the prefix
// keys and the L block keys of the row's own branch (block key j = the K/V
// row of src[b*L + j]), scale 1/sqrt(hd), all in fp32.
template <int HD>
__global__ void __launch_bounds__(256) attn_f32_kernel(const AttnF32 p) {
  constexpr int E = HD / 32;
  pdl_wait();
  pdl_trigger();
  const int n = min(max(p.n_dev[0], 0), p.R);
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int k = wid / p.n_q, h = wid - (wid / p.n_q) * p.n_q;
  if (k >= n) return;
  const int r = p.packed_idx[k];
  const int b = r / p.L;
  const int hk = h / p.g, hg = h - hk * p.g;
  const float* qrow = p.Q + ((static_cast<size_t>(hk) * p.R + k) * p.g + hg) * HD;
  float q[E], o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    q[e] = qrow[lane + 32 * e];
    o[e] = 0.f;
  }
  const float scale = 1.f / sqrtf(static_cast<float>(HD));
  float m = -INFINITY, l = 0.f;
  auto visit = [&](const float* krow, const float* vrow) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) s = fmaf(q[e], krow[lane + 32 * e], s);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    s *= scale;
    const float m_new = fmaxf(m, s);
    const float a = expf(m - m_new);  // 0 on the first key (m = -inf)
    const float pw = expf(s - m_new);
    l = l * a + pw;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = fmaf(pw, vrow[lane + 32 * e], o[e] * a);
    m = m_new;
  };
  for (int t = 0; t < p.P; ++t) {
    size_t tok = static_cast<size_t>(t);
    if (p.table) {
      const int page = p.table[t / p.page_size];
      if (page < 0 || page >= p.num_pages) {
        if (lane == 0) atomicOr(p.status, SPECFOLD_DEV_BAD_PAGE);
        continue;
      }
      tok = static_cast<size_t>(page) * p.page_size + t % p.page_size;
    }
    visit(p.pk + tok * p.k_ts + static_cast<size_t>(hk) * p.k_hs, p.pv + tok * p.v_ts + static_cast<size_t>(hk) * p.v_hs);
  }
  for (int j = 0; j < p.L; ++j) {
    const int s = p.src[b * p.L + j];
    if (s < 0 || s >= p.R) continue;
    const size_t off = (static_cast<size_t>(s) * p.n_kv + hk) * HD;
    visit(p.bK + off, p.bV + off);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* orow = p.O + static_cast<size_t>(k) * p.n_q * HD + static_cast<size_t>(h) * HD;
#pragma unroll
  for (int e = 0; e < E; ++e) orow[lane + 32 * e] = o[e] * inv;
}

}  // namespace

int launch_gemm_f32(const GemmCall& c, cudaStream_t st, const RowNorm* rn) {
  if (c.K <= 0 || c.K % kT || c.Mcap <= 0 || c.N <= 0 || c.N % kT) return SPECFOLD_EUNSUPPORTED;
  GemmF32 p;
  memset(&p, 0, sizeof(p));
  p.A = static_cast<const float*>(c.A);
  p.Mcap = c.Mcap;
  p.K = c.K;
  p.N = c.N;
  p.n_dev = c.n_dev;
  int col = 0;
  for (int j = 0; j < c.nb; ++j) {
    p.b[j] = static_cast<const float*>(c.b[j]);
    p.col0[j] = col;
    col += c.b_rows[j];
  }
  p.nb = c.nb;
  p.epi = c.epi;
  p.Y = static_cast<float*>(c.Y);
  p.ldy = c.ldy;
  p.resid = static_cast<const float*>(c.resid);
  p.ldr = c.ldr;
  p.row_idx = c.row_idx;
  p.Yk = static_cast<float*>(c.Yk);
  p.Yv = static_cast<float*>(c.Yv);
  p.n_q = c.n_q;
  p.n_kv = c.n_kv;
  p.hd = c.hd;
  p.g = c.n_kv > 0 ? c.n_q / c.n_kv : 1;
  p.R = c.Mcap;
  const dim3 grid(c.N / kT, (c.Mcap + kT - 1) / kT);
  launch_k(gemm_f32_kernel, grid, dim3(256), 0, st, p);
  count_launch();
  if (check_launch()) return SPECFOLD_ECUDA;
  if (c.epi == EPI_RESID_PACKED && rn)
    return launch_rmsnorm_rows(SPECFOLD_F32, c.Y, nullptr, c.n_dev, c.Mcap, c.N, rn->gain, rn->eps, rn->out, st);
  return SPECFOLD_OK;
}

int launch_attention_f32(const AttnCall& c, cudaStream_t st) {
  AttnF32 p;
  memset(&p, 0, sizeof(p));
  p.Q = static_cast<const float*>(c.Q);
  p.pk = static_cast<const float*>(c.pk.ptr);
  p.pv = static_cast<const float*>(c.pv.ptr);
  p.k_ts = c.pk.token_stride;
  p.k_hs = c.pk.head_stride;
  p.v_ts = c.pv.token_stride;
  p.v_hs = c.pv.head_stride;
  if (c.P > 0 && c.pk.block_table) {
    p.table = c.pk.block_table;
    p.page_size = c.pk.page_size;
    p.num_pages = std::min(c.pk.num_pages, c.pv.num_pages);
  }
  p.bK = static_cast<const float*>(c.blockK);
  p.bV = static_cast<const float*>(c.blockV);
  p.src = c.src;
  p.packed_idx = c.packed_idx;
  p.n_dev = c.n_dev;
  p.O = static_cast<float*>(c.O);
  p.P = c.P;
  p.L = c.L;
  p.R = c.B * c.L;
  p.n_q = c.n_q;
  p.n_kv = c.n_kv;
  p.g = c.n_q / c.n_kv;
  p.hd = c.hd;
  p.status = c.status;
  const int warps = p.R * c.n_q;
  const dim3 grid((warps + 7) / 8);
  if (c.hd == 128)
    launch_k(attn_f32_kernel<128>, grid, dim3(256), 0, st, p);
  else if (c.hd == 64)
    launch_k(attn_f32_kernel<64>, grid, dim3(256), 0, st, p);
  else
    return SPECFOLD_EUNSUPPORTED;
  count_launch();
  return check_launch();
}

}  // namespace sf
