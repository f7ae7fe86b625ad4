// Row-wise kernels of the folded layer: the residual gate (S1), provenance
// resolve + pack scan (S2, S3), the RMSNorm gathers (S3, S7) and the fold-fill
// of folded rows (S10).  All are HBM-bound: one warp per row, 16-byte
// vectorised coalesced loads, fp32 warp-shuffle reductions.
#include <algorithm>
#include <cstring>

#include "sf_device.cuh"
#include "sf_internal.h"

namespace sf {
namespace {

template <typename T>
struct VecT;
template <>
struct VecT<__nv_bfloat16> {
  static constexpr int N = 8;  // elements per 16-byte vector
  SF_DEV static void unpack(const uint4& u, float (&f)[8]) {
    f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
    f[4] = bf16lo(u.z); f[5] = bf16hi(u.z); f[6] = bf16lo(u.w); f[7] = bf16hi(u.w);
  }
  SF_DEV static uint4 pack(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
};
template <>
struct VecT<float> {
  static constexpr int N = 4;
  SF_DEV static void unpack(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  SF_DEV static uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

SF_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kRowWarps = 8;  // warps (rows) per block of the row kernels

// ------------------------------------------------------------------ S1 gate --
// One warp per row (b, i).  Child row and parent row are streamed once each
// (the parent row is shared by all its children and is normally an L2 hit).
template <typename T, int MAXV>
__global__ void __launch_bounds__(kRowWarps * 32)
gate_kernel(const T* __restrict__ H, const int32_t* __restrict__ parent, int B, int L, int d,
            float tau, uint8_t* __restrict__ fold, float* __restrict__ rel, uint8_t* __restrict__ fold_hist) {
  using V = VecT<T>;
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= B * L) return;
  const int b = row / L, i = row - b * L;
  const int nv = d / V::N;
  const uint4* c = reinterpret_cast<const uint4*>(H + static_cast<size_t>(row) * d);
  const int p = b > 0 ? parent[b] : -1;
  uint4 cv[MAXV], pv[MAXV];
  // the child row's first vectors do not depend on the parent index: they
  // are in flight while it arrives
  if (b > 0) {
#pragma unroll
    for (int u = 0; u < MAXV; ++u)
      if (lane + u * 32 < nv) cv[u] = __ldg(c + lane + u * 32);
  }
  if (b == 0 || p < 0 || p >= b) {  // root, or a parent the resolver will reject
    if (lane == 0) {
      fold[row] = 0;
      if (rel) rel[row] = -1.f;
      if (fold_hist) fold_hist[row] = 0;
    }
    return;
  }
  const uint4* q = reinterpret_cast<const uint4*>(H + (static_cast<size_t>(p) * L + i) * d);
  float num = 0.f, den = 0.f;
  for (int v0 = 0; v0 < nv; v0 += 32 * MAXV) {
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      const int v = v0 + lane + u * 32;
      if (v < nv) {
        if (v0 > 0) cv[u] = __ldg(c + v);
        pv[u] = __ldg(q + v);
      }
    }
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      const int v = v0 + lane + u * 32;
      if (v < nv) {
        float fc[V::N], fp[V::N];
        V::unpack(cv[u], fc);
        V::unpack(pv[u], fp);
#pragma unroll
        for (int e = 0; e < V::N; ++e) {
          const float df = fc[e] - fp[e];
          num = fmaf(df, df, num);
          den = fmaf(fp[e], fp[e], den);
        }
      }
    }
  }
  num = warp_sum(num);
  den = warp_sum(den);
  if (lane == 0) {
    const bool f = (num < tau * tau * den) || (num == 0.f && tau > 0.f);
    fold[row] = f ? 1 : 0;
    if (fold_hist) fold_hist[row] = f ? 1 : 0;
    if (rel) rel[row] = den > 0.f ? sqrtf(num / den) : (num == 0.f ? 0.f : __int_as_float(0x7f800000));
  }
}

// ------------------------------------------- S1 variant: gate vs source --
// One CTA per block position i.  Child (b, i) is compared with the row its
// parent's output at i comes from, s = src(parent[b], i), which depends on
// the parent's own decision: branches are processed level by level (a
// node's level is its number of hops to the root), each level's nodes in
// parallel, one warp per node, and the source branch of every decided node
// is kept in shared memory.  A parent outside [0, b) makes the row
// recompute (level 1), as in the parent gate.
template <typename T, int MAXV>
__global__ void __launch_bounds__(kRowWarps * 32)
gate_source_kernel(const T* __restrict__ H, const int32_t* __restrict__ parent, int B, int L, int d, float tau,
                   uint8_t* __restrict__ fold, float* __restrict__ rel, uint8_t* __restrict__ fold_hist) {
  using V = VecT<T>;
  extern __shared__ int sgs[];
  int* s_src = sgs;        // [B] branch whose row (., i) is reused
  int* s_lvl = sgs + B;    // [B]
  __shared__ int s_maxlvl;
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) s_maxlvl = 0;
  __syncthreads();
  for (int b = tid; b < B; b += blockDim.x) {
    int lv = 0, x = b;
    while (x > 0) {
      const int p = parent[x];
      ++lv;
      if (p < 0 || p >= x) break;
      x = p;
    }
    s_lvl[b] = lv;
    s_src[b] = b;
    atomicMax(&s_maxlvl, lv);
  }
  __syncthreads();
  if (tid == 0) {
    fold[i] = 0;
    if (rel) rel[i] = -1.f;
    if (fold_hist) fold_hist[i] = 0;
  }
  const int nv = d / V::N;
  for (int lv = 1; lv <= s_maxlvl; ++lv) {
    for (int b = w; b < B; b += kRowWarps) {
      if (s_lvl[b] != lv) continue;
      const int row = b * L + i;
      const int p = parent[b];
      if (p < 0 || p >= b) {
        if (lane == 0) {
          fold[row] = 0;
          if (rel) rel[row] = -1.f;
          if (fold_hist) fold_hist[row] = 0;
        }
        continue;  // s_src[b] stays b
      }
      const int sb = s_src[p];
      const uint4* c = reinterpret_cast<const uint4*>(H + static_cast<size_t>(row) * d);
      const uint4* q = reinterpret_cast<const uint4*>(H + (static_cast<size_t>(sb) * L + i) * d);
      float num = 0.f, den = 0.f;
      for (int v0 = 0; v0 < nv; v0 += 32 * MAXV) {
        uint4 cv[MAXV], pv[MAXV];
#pragma unroll
        for (int u = 0; u < MAXV; ++u) {
          const int v = v0 + lane + u * 32;
          if (v < nv) {
            cv[u] = __ldg(c + v);
            pv[u] = __ldg(q + v);
          }
        }
#pragma unroll
        for (int u = 0; u < MAXV; ++u) {
          const int v = v0 + lane + u * 32;
          if (v < nv) {
            float fc[V::N], fp[V::N];
            V::unpack(cv[u], fc);
            V::unpack(pv[u], fp);
#pragma unroll
            for (int e = 0; e < V::N; ++e) {
              const float df = fc[e] - fp[e];
              num = fmaf(df, df, num);
              den = fmaf(fp[e], fp[e], den);
            }
          }
        }
      }
      num = warp_sum(num);
      den = warp_sum(den);
      const bool f = (num < tau * tau * den) || (num == 0.f && tau > 0.f);
      if (lane == 0) {
        fold[row] = f ? 1 : 0;
        if (fold_hist) fold_hist[row] = f ? 1 : 0;
        if (rel) rel[row] = den > 0.f ? sqrtf(num / den) : (num == 0.f ? 0.f : __int_as_float(0x7f800000));
        s_src[b] = f ? sb : b;
      }
    }
    __syncthreads();  // this level's sources are visible to the next
  }
}

// ------------------------------------------------------- RMSNorm of a row --
// Gains of one row, for the norm: held in registers (GREG, loaded before the
// programmatic wait, overlapping the previous kernel) when the grid fits in
// one wave at one block per SM; otherwise read through L1 at the scaled
// store (every warp reads the same g), which keeps two or more blocks per SM.
template <typename T, int MAXV, bool GREG>
struct Gains {
  uint4 r[GREG ? MAXV : 1];
  const uint4* g;
  SF_DEV void load(const T* gp, int d, int lane) {
    g = reinterpret_cast<const uint4*>(gp);
    if constexpr (GREG) {
      const int nv = d / VecT<T>::N;
#pragma unroll
      for (int j = 0; j < MAXV; ++j)
        if (lane + 32 * j < nv) r[j] = __ldg(g + lane + 32 * j);
    }
  }
  SF_DEV uint4 at(int j, int vi) const {
    if constexpr (GREG) return r[j];
    return __ldg(g + vi);
  }
};

// y = x * g / sqrt(mean(x^2) + eps) for one row, one warp; the whole row is
// loaded before the reduction and held in registers until the scaled store.
// rawrow (optional) receives an unchanged copy of the row.
template <typename T, int MAXV, bool GREG>
SF_DEV void norm_row(const T* __restrict__ xrow, const Gains<T, MAXV, GREG>& gn, int d, float eps,
                     T* __restrict__ yrow, int lane, T* __restrict__ rawrow = nullptr) {
  using V = VecT<T>;
  const uint4* x = reinterpret_cast<const uint4*>(xrow);
  uint4* y = reinterpret_cast<uint4*>(yrow);
  const int nv = d / V::N;
  uint4 v[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < MAXV; ++j)
    if (lane + 32 * j < nv) v[j] = __ldg(x + lane + 32 * j);
  if (rawrow) {
    uint4* rw = reinterpret_cast<uint4*>(rawrow);
#pragma unroll
    for (int j = 0; j < MAXV; ++j)
      if (lane + 32 * j < nv) rw[lane + 32 * j] = v[j];
  }
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    if (lane + 32 * j < nv) {
      float f[V::N];
      V::unpack(v[j], f);
#pragma unroll
      for (int e = 0; e < V::N; ++e) ss = fmaf(f[e], f[e], ss);
    }
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / static_cast<float>(d) + eps);
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int vi = lane + 32 * j;
    if (vi < nv) {
      float f[V::N], gf[V::N];
      V::unpack(v[j], f);
      V::unpack(gn.at(j, vi), gf);
#pragma unroll
      for (int e = 0; e < V::N; ++e) f[e] = f[e] * inv * gf[e];
      y[vi] = V::pack(f);
    }
  }
}

// --------------------------------------------- S2 + S3 resolve / pack ------
// A row is recomputed iff fold[r] == 0, it is a root row, or its branch's
// parent is invalid (the chain cannot continue); src follows the fold chain
// through first parents to the recomputed row.  The packed list is the
// exclusive scan of the recomputed flags in row order.
//
// Every block recomputes the whole (cheap: R flags, short chains) resolve and
// scan in shared memory, writes its share of src / slot / packed_idx, and then
// gathers and RMS-normalises its eight packed rows -- so resolve, scan and the
// RMSNorm1 gather are one launch with no inter-block wait.
constexpr int kPackThreads = kRowWarps * 32;

// Branch whose row (., i) ends the fold chain that starts at (b, i), or -1
// when, without a parent table (pack alone), a folded non-root row is simply
// not recomputed.
SF_DEV int chain_end(const uint8_t* fold, const int32_t* parent, int b, int i, int L) {
  if (!parent) return (b > 0 && fold[b * L + i]) ? -1 : b;
  int s = b;
  while (s > 0 && fold[s * L + i]) {
    const int p = parent[s];
    if (p < 0 || p >= s) break;
    s = p;
  }
  return s;
}

template <typename T, int MAXV, bool GREG>
__global__ void __launch_bounds__(kPackThreads)
select_pack_kernel(const uint8_t* __restrict__ fold, const int32_t* __restrict__ parent, int B, int L,
                   int d, const T* __restrict__ H, const T* __restrict__ g1, float eps,
                   int32_t* __restrict__ src, int32_t* __restrict__ packed_idx, int32_t* __restrict__ slot,
                   int32_t* __restrict__ n_dev, T* __restrict__ X1, uint32_t* status,
                   int32_t* __restrict__ n_hist, int32_t* __restrict__ dep_rng, int32_t* __restrict__ dep_rows,
                   T* __restrict__ Xraw) {
  extern __shared__ int smem_i[];
  __shared__ int s_warp[kPackThreads / 32];
  __shared__ int s_bad;
  const int R = B * L;
  int* s_src = smem_i;          // [R] source row (-1: not recomputed, no source)
  int* s_slot = smem_i + R;     // [R] packed slot or -1
  int* s_inv = smem_i + 2 * R;  // [R + 1] row of packed slot k; block 0 reuses it for the dependents
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  Gains<T, MAXV, GREG> gn;
  if (X1) gn.load(g1, d, lane);  // weights: independent of earlier kernels
  pdl_wait();
  pdl_trigger();
  if (tid == 0) s_bad = 0;
  __syncthreads();
  if (blockIdx.x == 0)
    for (int b = tid; parent && b < B; b += kPackThreads) {
      const int p = parent[b];
      if ((b == 0 && p != -1) || (b > 0 && (p < 0 || p >= b))) atomicOr(&s_bad, 1);
    }
  const int ipt = (R + kPackThreads - 1) / kPackThreads;
  const int r0 = min(R, tid * ipt), r1 = min(R, r0 + ipt);
  // The chain walks are dependent loads: copy fold and parent into the
  // (not yet used) packed-slot array first, one coalesced pass, when they fit.
  const int fold_words = (R + 3) / 4;
  const bool staged = fold_words + (parent ? B : 0) <= R + 1;
  const uint8_t* fsrc = fold;
  const int32_t* psrc = parent;
  if (staged) {
    uint32_t* sf = reinterpret_cast<uint32_t*>(s_inv);
    for (int j = tid; j < fold_words; j += kPackThreads) {
      uint32_t wv = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (4 * j + e < R) wv |= static_cast<uint32_t>(fold[4 * j + e]) << (8 * e);
      sf[j] = wv;
    }
    if (parent)
      for (int b = tid; b < B; b += kPackThreads) s_inv[fold_words + b] = parent[b];
    __syncthreads();
    fsrc = reinterpret_cast<const uint8_t*>(s_inv);
    psrc = parent ? s_inv + fold_words : nullptr;
  }
  int cnt = 0;
  for (int r = r0; r < r1; ++r) {
    const int b = r / L, i = r - b * L;
    const int sb = chain_end(fsrc, psrc, b, i, L);
    const int sr = sb < 0 ? -1 : sb * L + i;
    s_src[r] = sr;
    cnt += (sr == r);
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[w] = incl;
  __syncthreads();
  if (w == 0) {
    int v = lane < kPackThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (lane < kPackThreads / 32) s_warp[lane] = v;  // inclusive warp totals
  }
  __syncthreads();
  const int n = s_warp[kPackThreads / 32 - 1];
  int off = (w > 0 ? s_warp[w - 1] : 0) + incl - cnt;
  for (int r = r0; r < r1; ++r) {
    if (s_src[r] == r) {
      s_slot[r] = off;
      s_inv[off] = r;
      ++off;
    } else {
      s_slot[r] = -1;
    }
  }
  __syncthreads();
  // this block's share of the global outputs
  const int chunk = (R + gridDim.x - 1) / gridDim.x;
  const int c0 = min(R, static_cast<int>(blockIdx.x) * chunk), c1 = min(R, c0 + chunk);
  for (int r = c0 + tid; r < c1; r += kPackThreads) {
    if (src) src[r] = s_src[r];
    if (slot) slot[r] = s_slot[r];
    if (packed_idx && s_slot[r] >= 0) packed_idx[s_slot[r]] = r;
  }
  if (blockIdx.x == 0 && tid == 0) {
    if (n_dev) n_dev[0] = n;
    if (n_hist) n_hist[0] = n;
    if (s_bad && status) atomicOr(status, SPECFOLD_DEV_BAD_PARENT);
  }
  const int k_norm = blockIdx.x * kRowWarps + w;
  const int r_norm = k_norm < n ? s_inv[k_norm] : -1;
  if (blockIdx.x == 0 && dep_rng) {
    // Block 0 groups the folded rows by the packed slot of their source
    // (counting sort in shared memory): for a recomputed row s,
    // dep_rows[dep_rng[2s] .. dep_rng[2s+1]) are the rows that take its output
    // plus their own difference.
    int* cnt = s_inv;  // [n + 1]
    __syncthreads();   // every read of s_inv above is done
    for (int k = tid; k <= n; k += kPackThreads) cnt[k] = 0;
    __syncthreads();
    for (int r = tid; r < R; r += kPackThreads) {
      const int sr = s_src[r];
      if (sr >= 0 && sr != r) atomicAdd(&cnt[s_slot[sr]], 1);
    }
    __syncthreads();
    // exclusive scan of cnt[0 .. n] (n + 1 entries) in place
    const int per = (n + 1 + kPackThreads - 1) / kPackThreads;
    const int c0 = min(n + 1, tid * per), c1 = min(n + 1, c0 + per);
    int loc = 0;
    for (int k = c0; k < c1; ++k) loc += cnt[k];
    int inc = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    __syncthreads();  // s_warp is free again
    if (lane == 31) s_warp[w] = inc;
    __syncthreads();
    if (w == 0) {
      int v = lane < kPackThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (lane < kPackThreads / 32) s_warp[lane] = v;
    }
    __syncthreads();
    int run = (w > 0 ? s_warp[w - 1] : 0) + inc - loc;
    for (int k = c0; k < c1; ++k) {
      const int c = cnt[k];
      cnt[k] = run;
      run += c;
    }
    __syncthreads();
    for (int r = tid; r < R; r += kPackThreads) {
      const int k = s_slot[r];
      if (k >= 0) reinterpret_cast<int2*>(dep_rng)[r] = make_int2(cnt[k], cnt[k + 1]);
    }
    __syncthreads();
    for (int r = tid; r < R; r += kPackThreads) {
      const int sr = s_src[r];
      if (sr >= 0 && sr != r) dep_rows[atomicAdd(&cnt[s_slot[sr]], 1)] = r;
    }
  }
  // RMSNorm1 gather of this block's packed rows (and, when asked, the rows
  // themselves)
  if (X1 && r_norm >= 0)
    norm_row<T, MAXV, GREG>(H + static_cast<size_t>(r_norm) * d, gn, d, eps, X1 + static_cast<size_t>(k_norm) * d,
                            lane, Xraw ? Xraw + static_cast<size_t>(k_norm) * d : nullptr);
}

// ------------------------------------------------------- RMSNorm rows --
// Y[k] = X[idx ? idx[k] : k] * g / sqrt(mean(X^2) + eps) for k < n.
template <typename T, int MAXV, bool GREG>
__global__ void __launch_bounds__(kRowWarps * 32)
rmsnorm_rows_kernel(const T* __restrict__ X, const int32_t* __restrict__ idx,
                    const int32_t* __restrict__ n_dev, int R, int d, const T* __restrict__ g,
                    float eps, T* __restrict__ Y) {
  const int k = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  Gains<T, MAXV, GREG> gn;
  if (k < R) gn.load(g, d, lane);  // weights: independent of earlier kernels
  pdl_wait();
  pdl_trigger();
  if (k >= R) return;
  const int n = n_dev ? min(max(n_dev[0], 0), R) : R;
  if (k >= n) return;
  const int r = idx ? idx[k] : k;
  norm_row<T, MAXV, GREG>(X + static_cast<size_t>(r) * d, gn, d, eps, Y + static_cast<size_t>(k) * d, lane);
}

// -------------------------------------------------------------- S10 fill --
template <typename T>
__global__ void __launch_bounds__(kRowWarps * 32)
fold_fill_kernel(const uint8_t* __restrict__ fold, const int32_t* __restrict__ src,
                 const T* __restrict__ Hin, T* __restrict__ Hout, int R, int d) {
  using V = VecT<T>;
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= R || !fold[r]) return;
  const int s = src[r];
  if (s == r || s < 0 || s >= R) return;
  const uint4* os = reinterpret_cast<const uint4*>(Hout + static_cast<size_t>(s) * d);
  const uint4* ir = reinterpret_cast<const uint4*>(Hin + static_cast<size_t>(r) * d);
  const uint4* is = reinterpret_cast<const uint4*>(Hin + static_cast<size_t>(s) * d);
  uint4* orow = reinterpret_cast<uint4*>(Hout + static_cast<size_t>(r) * d);
  const int nv = d / V::N;
  constexpr int U = 8;
  for (int v0 = lane; v0 < nv; v0 += 32 * U) {
    uint4 a[U], b[U], c[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < nv) {
        a[u] = os[v];
        b[u] = __ldg(ir + v);
        c[u] = __ldg(is + v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < nv) {
        float fa[V::N], fb[V::N], fc[V::N];
        V::unpack(a[u], fa);
        V::unpack(b[u], fb);
        V::unpack(c[u], fc);
#pragma unroll
        for (int e = 0; e < V::N; ++e) fa[e] = fa[e] + (fb[e] - fc[e]);
        orow[v] = V::pack(fa);
      }
    }
  }
}

// ------------------------------------------- variant sublayer helpers --
// Queries of every row for the literal attention correction: row r takes
// the query of its source row src[r] (packed slot slot[src[r]]).  One warp
// per (KV head, row) copies that row's g query heads (g*hd contiguous
// elements of the head-group-major layout).  Also writes the all-rows list
// (all_idx[r] = r, n_all = R) the attention and output projection then use.
template <typename T>
__global__ void __launch_bounds__(kRowWarps * 32)
gather_query_kernel(const T* __restrict__ Q, const int32_t* __restrict__ src, const int32_t* __restrict__ slot,
                    int R, int n_kv, int ghd, T* __restrict__ Qall, int32_t* __restrict__ all_idx,
                    int32_t* __restrict__ n_all) {
  pdl_wait();
  pdl_trigger();
  const int wid = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) n_all[0] = R;
  if (wid >= R * n_kv) return;
  const int h = wid / R, r = wid - h * R;
  if (h == 0 && lane == 0) all_idx[r] = r;
  const int s = src[r];
  const int k = (s >= 0 && s < R) ? slot[s] : -1;
  uint4* dst = reinterpret_cast<uint4*>(Qall + (static_cast<size_t>(h) * R + r) * ghd);
  const int nv = ghd * static_cast<int>(sizeof(T)) / 16;
  if (k < 0 || k >= R) {
    for (int v = lane; v < nv; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* from = reinterpret_cast<const uint4*>(Q + (static_cast<size_t>(h) * R + k) * ghd);
  for (int v = lane; v < nv; v += 32) dst[v] = from[v];
}

// Attention sublayer output of every row, in row order, from the packed
// rows: a recomputed row copies its packed row, a folded row r takes its
// source's plus its own input difference, Aall[r] = Ap[slot[s]] + (H[r] - H[s])
// (one rounding).  One warp per row.
template <typename T>
__global__ void __launch_bounds__(kRowWarps * 32)
unpack_fill_kernel(const T* __restrict__ Ap, const int32_t* __restrict__ src, const int32_t* __restrict__ slot,
                   const T* __restrict__ H, T* __restrict__ Aall, int R, int d) {
  using V = VecT<T>;
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= R) return;
  int s = src[r];
  if (s < 0 || s >= R) s = r;
  const int k = slot[s];
  uint4* orow = reinterpret_cast<uint4*>(Aall + static_cast<size_t>(r) * d);
  const int nv = d / V::N;
  if (k < 0 || k >= R) {
    for (int v = lane; v < nv; v += 32) orow[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* ap = reinterpret_cast<const uint4*>(Ap + static_cast<size_t>(k) * d);
  if (s == r) {
    for (int v = lane; v < nv; v += 32) orow[v] = ap[v];
    return;
  }
  const uint4* ir = reinterpret_cast<const uint4*>(H + static_cast<size_t>(r) * d);
  const uint4* is = reinterpret_cast<const uint4*>(H + static_cast<size_t>(s) * d);
  constexpr int U = 8;
  for (int v0 = lane; v0 < nv; v0 += 32 * U) {
    uint4 a[U], b[U], c[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < nv) {
        a[u] = ap[v];
        b[u] = __ldg(ir + v);
        c[u] = __ldg(is + v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < nv) {
        float fa[V::N], fb[V::N], fc[V::N];
        V::unpack(a[u], fa);
        V::unpack(b[u], fb);
        V::unpack(c[u], fc);
#pragma unroll
        for (int e = 0; e < V::N; ++e) fa[e] = fa[e] + (fb[e] - fc[e]);
        orow[v] = V::pack(fa);
      }
    }
  }
}

// ------------------------------------------------------------- S4b rope --
// One thread per (packed row, head, 8 rotation pairs).  Q: [n_kv][R*g][hd]
// (row k*g + j of KV head h holds query head h*g + j of packed row k);
// block keys: [R][n_kv][hd] at row packed_idx[k].  Frequencies are computed
// once per block in double and rounded to float; angles and sincosf in fp32.
SF_DEV void load8(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  x[0] = bf16lo(a.x); x[1] = bf16hi(a.x); x[2] = bf16lo(a.y); x[3] = bf16hi(a.y);
  x[4] = bf16lo(a.z); x[5] = bf16hi(a.z); x[6] = bf16lo(a.w); x[7] = bf16hi(a.w);
}
SF_DEV void load8(const float* p, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
SF_DEV void store8(__nv_bfloat16* p, const float (&y)[8]) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                            pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
}
SF_DEV void store8(float* p, const float (&y)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(y[0], y[1], y[2], y[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(y[4], y[5], y[6], y[7]);
}

template <typename T>
__global__ void __launch_bounds__(256)
rope_kernel(T* __restrict__ Q, T* __restrict__ Kb, const int32_t* __restrict__ packed_idx,
            const int32_t* __restrict__ n_dev, int R, int L, int P, int n_q, int n_kv, int hd, float theta) {
  __shared__ float s_freq[64];
  pdl_wait();
  pdl_trigger();
  const int half = hd / 2;
  for (int j = threadIdx.x; j < half; j += blockDim.x)
    s_freq[j] = static_cast<float>(pow(static_cast<double>(theta), -2.0 * j / hd));
  __syncthreads();
  const int n = min(max(n_dev[0], 0), R);
  const int g = n_q / n_kv;
  const int heads = n_q + n_kv;
  const int G8 = half / 8;
  const long long total = static_cast<long long>(n) * heads * G8;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(idx / (heads * G8));
    const int rem = static_cast<int>(idx - static_cast<long long>(k) * heads * G8);
    const int h = rem / G8;
    const int j0 = (rem - h * G8) * 8;
    const int r = packed_idx[k];
    if (r < 0 || r >= R) continue;
    const float pos = static_cast<float>(P + r % L);
    T* row;
    if (h < n_q) {
      const int hk = h / g, hg = h - hk * g;
      row = Q + ((static_cast<size_t>(hk) * R + k) * g + hg) * hd;
    } else {
      row = Kb + (static_cast<size_t>(r) * n_kv + (h - n_q)) * hd;
    }
    float x1[8], x2[8], y1[8], y2[8];
    load8(row + j0, x1);
    load8(row + half + j0, x2);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float sn, cs;
      sincosf(pos * s_freq[j0 + e], &sn, &cs);
      y1[e] = x1[e] * cs - x2[e] * sn;
      y2[e] = x2[e] * cs + x1[e] * sn;
    }
    store8(row + j0, y1);
    store8(row + half + j0, y2);
  }
}

// ------------------------------------------------ S1 + S2 + S3 fused --
// One launch for the gate, the resolve and the pack of the parent-gate
// layer, on a grid of at most one CTA per SM (all resident at once).
//
// Phase 1 (gate): CTA j owns the contiguous rows [j*chunk, (j+1)*chunk), one
// warp per row.  Each row streams its child and parent rows once, decides
// fold (squared comparison, as the standalone gate) and, for RMSNorm1, sums
// the squares of the child row; with HOLD (at most one row per warp) the row
// stays in registers until its packed slot is known.  The CTA publishes its
// count of recomputed rows.
// Grid barrier (bounded, see grid_barrier).
// Phase 2 (pack): every CTA stages all R decisions in shared memory; its
// rows' packed slots follow from the counts of the CTAs before it and a
// local scan (branch-major, position-ascending order); it writes src (fold
// chains walked in shared memory), slot, packed_idx and X1 of its recomputed
// rows.  A fold chain never leaves its block position, so the folded rows are
// grouped by source per position: CTA j groups positions j, j + G, ...; the
// folded rows of position i occupy dep_rows[i*B .. (i+1)*B).
constexpr int kGPWarps = 16;
constexpr int kGPThreads = kGPWarps * 32;
constexpr int kGPMaxCtas = 256;
constexpr int kGPPass = 8;  // vectors per lane per pass without HOLD

struct GatePackArgs {
  const void* H;
  const int32_t* parent;
  int B, L, d;
  float tau;
  const void* g1;
  float eps;
  uint8_t* fold;
  float* rel;
  uint8_t* fold_hist;
  int32_t* src;
  int32_t* packed_idx;
  int32_t* slot;
  int32_t* n_dev;
  int32_t* n_hist;
  void* X1;
  int32_t* dep_rng;
  int32_t* dep_rows;
  uint32_t* bar;
  int32_t* cta_cnt;
  uint32_t* status;
  int chunk;   // rows per CTA
  int batch;   // rows per shared-memory batch
};

// Exclusive prefix sums of v[0 .. N) into out (may alias v); returns the
// total.  Called by every thread of the block; s_warp holds 32 ints.
SF_DEV int block_scan_excl(const int* v, int* out, int N, int* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int b0 = min(N, tid * per), b1 = min(N, b0 + per);
  int loc = 0;
  for (int k = b0; k < b1; ++k) loc += v[k];
  int inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) s_warp[w] = inc;
  __syncthreads();
  if (w == 0) {
    int x = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += t;
    }
    if (lane < nw) s_warp[lane] = x;
  }
  __syncthreads();
  int run = (w > 0 ? s_warp[w - 1] : 0) + inc - loc;
  const int total = s_warp[nw - 1];
  for (int k = b0; k < b1; ++k) {
    const int c = v[k];
    out[k] = run;
    run += c;
  }
  __syncthreads();
  return total;
}

// Branch at the end of the fold chain that starts at (b, i), on staged
// decisions: a folded row always has a valid parent.
SF_DEV int chain_end_smem(const uint8_t* f, const int* par, int b, int i, int L, int B) {
  int s = b;
  for (int hop = 0; hop < B && s > 0 && f[s * L + i]; ++hop) s = par[s];
  return s;
}

// The dependents lists of block position i for a draft graph of at most 32
// branches, in one warp (lane b = branch b): the same outputs as the block
// loop at the end of gate_pack_kernel, with each source's folded rows in
// ascending branch order.
SF_DEV void deps_warp(const GatePackArgs& a, const uint8_t* f, const int* par, int i, int L, int B, int lane) {
  const bool on = lane < B;
  const int sb = on ? (f[lane * L + i] ? chain_end_smem(f, par, lane, i, L, B) : lane) : -1;
  const unsigned grp = __match_any_sync(0xffffffffu, sb);  // lanes that share this source
  const bool is_src = on && sb == lane;
  const int cnt = is_src ? __popc(grp) - 1 : 0;
  int inc = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  const int start = inc - cnt;  // first slot of this source's group
  if (is_src) reinterpret_cast<int2*>(a.dep_rng)[lane * L + i] = make_int2(i * B + start, i * B + start + cnt);
  const int sstart = __shfl_sync(0xffffffffu, start, on ? sb : 0);
  if (on && !is_src) {
    const int rank = __popc(grp & ((1u << lane) - 1u) & ~(1u << sb));
    a.dep_rows[i * B + sstart + rank] = lane * L + i;
  }
}

template <typename T>
SF_DEV void accum_gate(const uint4& c, const uint4& q, float& num, float& den) {
  using V = VecT<T>;
  float fc[V::N], fp[V::N];
  V::unpack(c, fc);
  V::unpack(q, fp);
#pragma unroll
  for (int e = 0; e < V::N; ++e) {
    const float df = fc[e] - fp[e];
    num = fmaf(df, df, num);
    den = fmaf(fp[e], fp[e], den);
  }
}

template <typename T>
SF_DEV void accum_sq(const uint4& c, float& ss) {
  using V = VecT<T>;
  float f[V::N];
  V::unpack(c, f);
#pragma unroll
  for (int e = 0; e < V::N; ++e) ss = fmaf(f[e], f[e], ss);
}

template <typename T>
SF_DEV uint4 scale_vec(const uint4& x, const uint4& g, float inv) {
  using V = VecT<T>;
  float f[V::N], gf[V::N];
  V::unpack(x, f);
  V::unpack(g, gf);
#pragma unroll
  for (int e = 0; e < V::N; ++e) f[e] = f[e] * inv * gf[e];
  return V::pack(f);
}

// Gate decision of one row from its sums (the standalone gate's rule).
SF_DEV void gate_write(const GatePackArgs& a, int row, bool valid, float num, float den) {
  const bool f = valid && ((num < a.tau * a.tau * den) || (num == 0.f && a.tau > 0.f));
  a.fold[row] = f ? 1 : 0;
  if (a.fold_hist) a.fold_hist[row] = f ? 1 : 0;
  if (a.rel)
    a.rel[row] = !valid ? -1.f : (den > 0.f ? sqrtf(num / den) : (num == 0.f ? 0.f : __int_as_float(0x7f800000)));
}

template <typename T, int MAXV, bool HOLD>
__global__ void __launch_bounds__(kGPThreads, 1) gate_pack_kernel(const __grid_constant__ GatePackArgs a) {
  using V = VecT<T>;
  extern __shared__ __align__(128) uint8_t gp_smem[];
  __shared__ int s_warp[32];
  __shared__ int s_nb, s_n, s_bad;
  __shared__ volatile int s_flag;
  __shared__ volatile int s_abort;
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ __align__(8) uint64_t s_gbar;  // the gains' copy
  const int B = a.B, L = a.L, d = a.d, R = B * L;
  const int nv = d / V::N;  // 16-byte vectors per row
  const uint32_t rowb = static_cast<uint32_t>(d) * sizeof(T);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  // shared memory: rows [batch][nv] | gains [nv] | parent [B] | decisions [R, 16-rounded] | three int arrays
  uint4* s_rows = reinterpret_cast<uint4*>(gp_smem);
  uint4* s_g = s_rows + static_cast<size_t>(a.batch) * nv;
  int* s_par = reinterpret_cast<int*>(s_g + nv);
  uint8_t* s_fold = reinterpret_cast<uint8_t*>(s_par + ((B + 3) & ~3));
  int* s_c1 = reinterpret_cast<int*>(s_fold + ((R + 15) & ~15));  // [max(B, chunk)]
  int* s_c2 = s_c1 + max(B, a.chunk);                              // [B]
  int* s_c3 = s_c2 + B;                                            // [B]
  const uint32_t bar = smem_u32(&s_bar), gbar = smem_u32(&s_gbar);
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(gbar, 1);
    fence_mbar_init();
    s_abort = 0;
    s_bad = 0;
    // gains: weights, independent of earlier kernels; needed only by the
    // RMSNorm after the grid barrier, so nothing waits for them until then
    mbar_arrive_expect_tx(gbar, rowb);
    bulk_load(smem_u32(s_g), a.g1, rowb, gbar);
  }
  pdl_wait();
  __syncthreads();

  // ---------------------------------------------------- phase 1: gate --
  const int c0 = blockIdx.x * a.chunk, c1 = min(R, c0 + a.chunk);
  const int nch = max(c1 - c0, 0);
  const T* H = static_cast<const T*>(a.H);
  float ss_hold = 0.f;
  int act_here = 0;     // recomputed rows of this warp (lane 0)
  int issued_bt = -1;   // last batch whose copies were issued (thread 0)
  for (int bt = 0; bt * a.batch < nch; ++bt) {
    const int r0 = c0 + bt * a.batch, nr = min(a.batch, c1 - r0);
    if (bt > 0) {
      __syncthreads();  // the previous batch's rows are consumed
      if (s_abort) break;
    }
    if (tid == 0) {
      issued_bt = bt;
      // the child rows of this batch, one bulk copy each
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nr) * rowb);
      for (int t = 0; t < nr; ++t)
        bulk_load(smem_u32(s_rows + static_cast<size_t>(t) * nv), H + static_cast<size_t>(r0 + t) * d, rowb, bar);
    }
    for (int t = w; t < nr; t += kGPWarps) {
      const int r = r0 + t;
      const int b = r / L, i = r - b * L;
      const int p = b > 0 ? __ldg(a.parent + b) : -1;
      const bool valid = b > 0 && p >= 0 && p < b;
      // the parent row (usually an L2 hit) into registers while the child
      // rows stream into shared memory
      const uint4* q = reinterpret_cast<const uint4*>(H + (static_cast<size_t>(valid ? p : 0) * L + i) * d);
      uint4 pv[MAXV];
      if (valid) {
#pragma unroll
        for (int u = 0; u < MAXV; ++u)
          if (lane + 32 * u < nv) pv[u] = __ldg(q + lane + 32 * u);
      }
      if (!mbar_wait(bar, bt & 1, &s_abort, a.status, kWaitLimitNs, kSiteGpRows)) break;
      const uint4* c = s_rows + static_cast<size_t>(t) * nv;
      float num = 0.f, den = 0.f, ss = 0.f;
#pragma unroll
      for (int u = 0; u < MAXV; ++u) {
        const int v = lane + 32 * u;
        if (v < nv) {
          const uint4 cv = c[v];
          if (valid) accum_gate<T>(cv, pv[u], num, den);
          accum_sq<T>(cv, ss);
        }
      }
      num = warp_sum(num);
      den = warp_sum(den);
      const bool f = valid && ((num < a.tau * a.tau * den) || (num == 0.f && a.tau > 0.f));
      if (lane == 0) {
        gate_write(a, r, valid, num, den);
        act_here += f ? 0 : 1;
      }
      if constexpr (HOLD) ss_hold = warp_sum(ss);
    }
  }
  // the draft graph, for the pack (and its validity, once)
  for (int b = tid; b < B; b += kGPThreads) {
    const int p = a.parent[b];
    s_par[b] = p;
    if ((b == 0 && p != -1) || (b > 0 && (p < 0 || p >= b))) s_bad = 1;
  }
  // this CTA's count of recomputed rows
  if (lane == 0) s_warp[w] = act_here;
  __syncthreads();
  if (s_abort) {  // a copy never landed: give the last ones a short bound, then leave
    if (tid == 0) {
      int never = 0;
      if (issued_bt >= 0) mbar_wait(bar, issued_bt & 1, &never, nullptr, 10000000ull);
      mbar_wait(gbar, 0, &never, nullptr, 10000000ull);
    }
    return;
  }
  if (tid == 0) {
    int t = 0;
    for (int j = 0; j < kGPWarps; ++j) t += s_warp[j];
    a.cta_cnt[blockIdx.x] = t;
    if (blockIdx.x == 0 && s_bad && a.status) atomicOr(a.status, SPECFOLD_DEV_BAD_PARENT);
  }
  if (!grid_barrier(a.bar, a.status, &s_flag)) {
    if (tid == 0) {  // the gains' copy targets this CTA's shared memory
      int never = 0;
      mbar_wait(gbar, 0, &never, nullptr, 10000000ull);
    }
    return;
  }
  pdl_trigger();

  // ---------------------------------------------------- phase 2: pack --
  {
    const uint4* fg = reinterpret_cast<const uint4*>(a.fold);
    uint4* fs = reinterpret_cast<uint4*>(s_fold);
    for (int j = tid; j < (R + 15) / 16; j += kGPThreads) fs[j] = __ldcg(fg + j);
  }
  if (w == 0) {
    int tot = 0, before = 0;
    for (int j = lane; j < static_cast<int>(gridDim.x); j += 32) {
      const int v = __ldcg(a.cta_cnt + j);
      tot += v;
      before += j < static_cast<int>(blockIdx.x) ? v : 0;
    }
    tot = __reduce_add_sync(0xffffffffu, tot);
    before = __reduce_add_sync(0xffffffffu, before);
    if (lane == 0) {
      s_n = tot;
      s_nb = before;
    }
  }
  __syncthreads();
  const int n = s_n, nb = s_nb;
  for (int t = tid; t < nch; t += kGPThreads) s_c1[t] = s_fold[c0 + t] ? 0 : 1;
  __syncthreads();
  block_scan_excl(s_c1, s_c1, nch, s_warp);  // local rank of each recomputed row
  for (int t = tid; t < nch; t += kGPThreads) {
    const int r = c0 + t;
    const int b = r / L, i = r - b * L;
    const bool act = !s_fold[r];
    const int k = nb + s_c1[t];
    a.slot[r] = act ? k : -1;
    if (act) a.packed_idx[k] = r;
    a.src[r] = act ? r : chain_end_smem(s_fold, s_par, b, i, L, B) * L + i;
  }
  if (blockIdx.x == 0 && tid == 0) {
    a.n_dev[0] = n;
    if (a.n_hist) a.n_hist[0] = n;
  }
  // with at most 32 branches and a warp to spare, the last warp builds the
  // dependents lists of this CTA's block positions while the others write X1
  const bool deps_by_warp = a.dep_rng && HOLD && B <= 32 && nch < kGPWarps;
  if (deps_by_warp && w == kGPWarps - 1)
    for (int i = blockIdx.x; i < L; i += gridDim.x) deps_warp(a, s_fold, s_par, i, L, B, lane);
  // RMSNorm1 of this CTA's recomputed rows: X1[k] = H[r] * g1 / rms(H[r])
  T* X1 = static_cast<T*>(a.X1);
  if constexpr (HOLD) {
    const int r = c0 + w;
    if (w < nch && !s_fold[r] && mbar_wait(gbar, 0, &s_abort, a.status, kWaitLimitNs, kSiteGpGains)) {
      const float inv = rsqrtf(ss_hold / static_cast<float>(d) + a.eps);
      const uint4* x = s_rows + static_cast<size_t>(w) * nv;
      uint4* y = reinterpret_cast<uint4*>(X1 + static_cast<size_t>(nb + s_c1[w]) * d);
      for (int v = lane; v < nv; v += 32) y[v] = scale_vec<T>(x[v], s_g[v], inv);
    }
  } else {
    const bool g_ok = mbar_wait(gbar, 0, &s_abort, a.status, kWaitLimitNs, kSiteGpGains);
    for (int t = w; t < nch && g_ok; t += kGPWarps) {
      const int r = c0 + t;
      if (s_fold[r]) continue;
      const uint4* x = reinterpret_cast<const uint4*>(H + static_cast<size_t>(r) * d);
      float ss = 0.f;
      for (int v0 = 0; v0 < nv; v0 += 32 * kGPPass) {
        uint4 xv[kGPPass];
#pragma unroll
        for (int u = 0; u < kGPPass; ++u)
          if (v0 + lane + 32 * u < nv) xv[u] = __ldg(x + v0 + lane + 32 * u);
#pragma unroll
        for (int u = 0; u < kGPPass; ++u)
          if (v0 + lane + 32 * u < nv) accum_sq<T>(xv[u], ss);
      }
      const float inv = rsqrtf(warp_sum(ss) / static_cast<float>(d) + a.eps);
      uint4* y = reinterpret_cast<uint4*>(X1 + static_cast<size_t>(nb + s_c1[t]) * d);
      for (int v = lane; v < nv; v += 32) y[v] = scale_vec<T>(__ldg(x + v), s_g[v], inv);
    }
  }
  if (deps_by_warp || !a.dep_rng) return;  // lists built, or not asked for
  // folded rows grouped by source, one block position at a time
  for (int i = blockIdx.x; i < L; i += gridDim.x) {
    __syncthreads();  // the arrays are free again
    for (int b = tid; b < B; b += kGPThreads) s_c2[b] = 0;
    __syncthreads();
    for (int b = tid; b < B; b += kGPThreads) {
      const int sb = s_fold[b * L + i] ? chain_end_smem(s_fold, s_par, b, i, L, B) : b;
      s_c1[b] = sb;
      if (sb != b) atomicAdd(&s_c2[sb], 1);
    }
    __syncthreads();
    block_scan_excl(s_c2, s_c3, B, s_warp);  // s_c3: first slot of each source's group
    for (int b = tid; b < B; b += kGPThreads)
      if (s_c1[b] == b)
        reinterpret_cast<int2*>(a.dep_rng)[b * L + i] = make_int2(i * B + s_c3[b], i * B + s_c3[b] + s_c2[b]);
    __syncthreads();
    for (int b = tid; b < B; b += kGPThreads) {
      const int sb = s_c1[b];
      if (sb != b) a.dep_rows[i * B + atomicAdd(&s_c3[sb], 1)] = b * L + i;
    }
  }
}

// ------------------------------------------------------ bounded-wait probe --
__global__ void timeout_probe_kernel(uint32_t* status, uint64_t wait_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing arrives on this barrier: the wait has to run out.
    mbar_wait(smem_u32(&bar), 0, &abort_flag, status, wait_ns, kSiteProbe);
  }
  __syncthreads();
}

}  // namespace

int launch_rope(int dtype, void* Q, void* Kb, const int32_t* packed_idx, const int32_t* n_dev, int R, int L, int P,
                int n_q, int n_kv, int hd, float theta, cudaStream_t st) {
  const long long total = static_cast<long long>(R) * (n_q + n_kv) * (hd / 16);
  const int grid = std::max(static_cast<int>(std::min<long long>((total + 255) / 256, 8LL * num_sms())), 1);
  if (dtype == SPECFOLD_BF16)
    launch_k(rope_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st, static_cast<__nv_bfloat16*>(Q),
             static_cast<__nv_bfloat16*>(Kb), packed_idx, n_dev, R, L, P, n_q, n_kv, hd, theta);
  else
    launch_k(rope_kernel<float>, dim3(grid), dim3(256), 0, st, static_cast<float*>(Q), static_cast<float*>(Kb),
             packed_idx, n_dev, R, L, P, n_q, n_kv, hd, theta);
  count_launch();
  return check_launch();
}

int launch_gate(int dtype, const void* H, const int32_t* parent, int B, int L, int d, float tau,
                uint8_t* fold, float* rel, cudaStream_t st, uint8_t* fold_hist) {
  const int R = B * L;
  const dim3 grid((R + kRowWarps - 1) / kRowWarps), block(kRowWarps * 32);
  // A whole row in flight per lane (one pass) needs one block per SM; when
  // the grid would then take more than one wave, two passes of eight
  // vectors keep two blocks per SM instead.
  int per_lane = (d / (dtype == SPECFOLD_BF16 ? 8 : 4) + 31) / 32;
  if (static_cast<int>(grid.x) > num_sms()) per_lane = std::min(per_lane, 8);
  if (dtype == SPECFOLD_BF16) {
    const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(H);
    if (per_lane <= 8)
      launch_k(gate_kernel<__nv_bfloat16, 8>, dim3(grid), dim3(block), 0, st, h, parent, B, L, d, tau, fold, rel, fold_hist);
    else
      launch_k(gate_kernel<__nv_bfloat16, 16>, dim3(grid), dim3(block), 0, st, h, parent, B, L, d, tau, fold, rel, fold_hist);
  } else {
    const float* h = static_cast<const float*>(H);
    if (per_lane <= 8)
      launch_k(gate_kernel<float, 8>, dim3(grid), dim3(block), 0, st, h, parent, B, L, d, tau, fold, rel, fold_hist);
    else
      launch_k(gate_kernel<float, 16>, dim3(grid), dim3(block), 0, st, h, parent, B, L, d, tau, fold, rel, fold_hist);
  }
  count_launch();
  return check_launch();
}

size_t gate_pack_sync_bytes() { return 128 + sizeof(int32_t) * kGPMaxCtas; }

constexpr int kGPMaxSmem = 200 * 1024;  // the launcher's bound on the kernel's dynamic shared memory

template <typename T, int MAXV, bool HOLD>
static int gate_pack_go(const GatePackArgs& a, int grid, size_t smem, cudaStream_t st) {
  // the limit is raised once per device, to the largest size any shape asks for
  if (smem > 48 * 1024)
    if (const int rc = smem_limit_once(gate_pack_kernel<T, MAXV, HOLD>, kGPMaxSmem)) return rc;
  launch_k(gate_pack_kernel<T, MAXV, HOLD>, dim3(grid), dim3(kGPThreads), smem, st, a);
  count_launch();
  return check_launch();
}

int launch_gate_pack(int dtype, const void* H, const int32_t* parent, int B, int L, int d, float tau,
                     const void* g1, float eps, uint8_t* fold, float* rel, int32_t* src, int32_t* packed_idx,
                     int32_t* slot, int32_t* n_dev, void* X1, int32_t* dep_rng, int32_t* dep_rows, void* sync,
                     uint32_t* status, cudaStream_t st, uint8_t* fold_hist, int32_t* n_hist) {
  const int R = B * L;
  const int es = dtype == SPECFOLD_BF16 ? 2 : 4;
  const int nv = d * es / 16;
  const int per_lane = (nv + 31) / 32;
  const int sms = std::max(1, std::min(num_sms(), kGPMaxCtas));
  const int chunk = (R + sms - 1) / sms;
  const int grid = (R + chunk - 1) / chunk;
  // child rows staged in shared memory: up to 16 rows, 128 KB
  const size_t rowb = static_cast<size_t>(d) * es;
  const int batch = static_cast<int>(std::max<size_t>(1, std::min<size_t>(kGPWarps, (128u << 10) / rowb)));
  const size_t smem = static_cast<size_t>(batch) * rowb + static_cast<size_t>(nv) * 16 +
                      4 * static_cast<size_t>((B + 3) & ~3) + ((R + 15) & ~15) +
                      4 * static_cast<size_t>(std::max(B, chunk)) + 8 * static_cast<size_t>(B);
  if (per_lane > 16 || smem > static_cast<size_t>(kGPMaxSmem)) return SPECFOLD_EUNSUPPORTED;
  GatePackArgs a;
  memset(&a, 0, sizeof(a));
  a.H = H;
  a.parent = parent;
  a.B = B;
  a.L = L;
  a.d = d;
  a.tau = tau;
  a.g1 = g1;
  a.eps = eps;
  a.fold = fold;
  a.rel = rel;
  a.fold_hist = fold_hist;
  a.src = src;
  a.packed_idx = packed_idx;
  a.slot = slot;
  a.n_dev = n_dev;
  a.n_hist = n_hist;
  a.X1 = X1;
  a.dep_rng = dep_rng;
  a.dep_rows = dep_rows;
  a.bar = static_cast<uint32_t*>(sync);
  a.cta_cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(sync) + 128);
  a.status = status;
  a.chunk = chunk;
  a.batch = batch;
  // the whole chunk stays staged for RMSNorm1 (one row per warp), or the
  // rows are read again from L2 after the barrier
  const bool hold = chunk <= batch;
#define SF_GP(TT)                                                                          \
  if (per_lane <= 4) return hold ? gate_pack_go<TT, 4, true>(a, grid, smem, st)           \
                                 : gate_pack_go<TT, 4, false>(a, grid, smem, st);         \
  if (per_lane <= 8) return hold ? gate_pack_go<TT, 8, true>(a, grid, smem, st)           \
                                 : gate_pack_go<TT, 8, false>(a, grid, smem, st);         \
  return hold ? gate_pack_go<TT, 16, true>(a, grid, smem, st) : gate_pack_go<TT, 16, false>(a, grid, smem, st)
  if (dtype == SPECFOLD_BF16) {
    SF_GP(__nv_bfloat16);
  }
  SF_GP(float);
#undef SF_GP
}

int launch_gate_source(int dtype, const void* H, const int32_t* parent, int B, int L, int d, float tau,
                       uint8_t* fold, float* rel, cudaStream_t st, uint8_t* fold_hist) {
  const size_t smem = static_cast<size_t>(2) * B * sizeof(int);
  const int per_lane = (d / (dtype == SPECFOLD_BF16 ? 8 : 4) + 31) / 32;
  auto prep = [&](auto kern, int) -> bool {
    if (smem <= 48 * 1024) return true;
    return smem_limit_once(kern, 2 * SPECFOLD_MAX_ROWS * static_cast<int>(sizeof(int))) == SPECFOLD_OK;
  };
  const dim3 grid(L), block(kRowWarps * 32);
  if (dtype == SPECFOLD_BF16) {
    const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(H);
    if (per_lane <= 8) {
      if (!prep(gate_source_kernel<__nv_bfloat16, 8>, 0)) return SPECFOLD_ECUDA;
      launch_k(gate_source_kernel<__nv_bfloat16, 8>, grid, block, smem, st, h, parent, B, L, d, tau, fold, rel,
               fold_hist);
    } else {
      if (!prep(gate_source_kernel<__nv_bfloat16, 16>, 1)) return SPECFOLD_ECUDA;
      launch_k(gate_source_kernel<__nv_bfloat16, 16>, grid, block, smem, st, h, parent, B, L, d, tau, fold, rel,
               fold_hist);
    }
  } else {
    const float* h = static_cast<const float*>(H);
    if (per_lane <= 8) {
      if (!prep(gate_source_kernel<float, 8>, 2)) return SPECFOLD_ECUDA;
      launch_k(gate_source_kernel<float, 8>, grid, block, smem, st, h, parent, B, L, d, tau, fold, rel, fold_hist);
    } else {
      if (!prep(gate_source_kernel<float, 16>, 3)) return SPECFOLD_ECUDA;
      launch_k(gate_source_kernel<float, 16>, grid, block, smem, st, h, parent, B, L, d, tau, fold, rel, fold_hist);
    }
  }
  count_launch();
  return check_launch();
}

template <typename T, int MAXV, bool GREG>
static int select_pack_launch(const uint8_t* fold, const int32_t* parent, int B, int L, int d, const void* H,
                              const void* g1, float eps, int32_t* src, int32_t* packed_idx, int32_t* slot,
                              int32_t* n_dev, void* X1, uint32_t* status, cudaStream_t st, int32_t* n_hist, int32_t* dep_rng,
                              int32_t* dep_rows, void* Xraw) {
  const int R = B * L;
  const size_t smem = (static_cast<size_t>(3) * R + 1) * sizeof(int);
  if (smem > 48 * 1024 &&
      smem_limit_once(select_pack_kernel<T, MAXV, GREG>, (3 * SPECFOLD_MAX_ROWS + 1) * static_cast<int>(sizeof(int))))
    return SPECFOLD_ECUDA;
  const dim3 grid((R + kRowWarps - 1) / kRowWarps), block(kPackThreads);
  launch_k(select_pack_kernel<T, MAXV, GREG>, dim3(grid), dim3(block), smem, st, fold, parent, B, L, d, static_cast<const T*>(H),
                                                          static_cast<const T*>(g1), eps, src, packed_idx, slot,
                                                          n_dev, static_cast<T*>(X1), status, n_hist, dep_rng, dep_rows,
                                                          static_cast<T*>(Xraw));
  count_launch();
  return check_launch();
}

template <typename T>
static int select_pack_dispatch(const uint8_t* fold, const int32_t* parent, int B, int L, int d, const void* H,
                                const void* g1, float eps, int32_t* src, int32_t* packed_idx, int32_t* slot,
                                int32_t* n_dev, void* X1, uint32_t* status, cudaStream_t st, int32_t* n_hist, int32_t* dep_rng,
                                int32_t* dep_rows, void* Xraw) {
  const int per_lane = X1 ? (d / VecT<T>::N + 31) / 32 : 1;
  // gains in registers when the grid fits one wave at one block per SM
  const bool greg = (B * L + kRowWarps - 1) / kRowWarps <= num_sms();
#define SF_SP(MV)                                                                                                 \
  return greg ? select_pack_launch<T, MV, true>(fold, parent, B, L, d, H, g1, eps, src, packed_idx, slot, n_dev,  \
                                                X1, status, st, n_hist, dep_rng, dep_rows, Xraw)                  \
              : select_pack_launch<T, MV, false>(fold, parent, B, L, d, H, g1, eps, src, packed_idx, slot, n_dev, \
                                                 X1, status, st, n_hist, dep_rng, dep_rows, Xraw)
  if (per_lane <= 4) SF_SP(4);
  if (per_lane <= 8) SF_SP(8);
  if (per_lane <= 16) SF_SP(16);
  if (per_lane <= 32) SF_SP(32);
#undef SF_SP
  return SPECFOLD_EUNSUPPORTED;
}

int launch_select_pack(int dtype, const uint8_t* fold, const int32_t* parent, int B, int L, int d, const void* H,
                       const void* g1, float eps, int32_t* src, int32_t* packed_idx, int32_t* slot, int32_t* n_dev,
                       void* X1, uint32_t* status, cudaStream_t st, int32_t* n_hist, int32_t* dep_rng,
                       int32_t* dep_rows, void* Xraw) {
  if (Xraw && !X1) return SPECFOLD_EINVAL;
  if (dtype == SPECFOLD_BF16)
    return select_pack_dispatch<__nv_bfloat16>(fold, parent, B, L, d, H, g1, eps, src, packed_idx, slot, n_dev, X1,
                                               status, st, n_hist, dep_rng, dep_rows, Xraw);
  return select_pack_dispatch<float>(fold, parent, B, L, d, H, g1, eps, src, packed_idx, slot, n_dev, X1, status,
                                     st, n_hist, dep_rng, dep_rows, Xraw);
}

template <typename T>
static void rmsnorm_dispatch(const void* X, const int32_t* idx, const int32_t* n_dev, int R, int d, const void* g,
                             float eps, void* Y, cudaStream_t st) {
  const dim3 grid((R + kRowWarps - 1) / kRowWarps), block(kRowWarps * 32);
  const int per_lane = (d / VecT<T>::N + 31) / 32;
  const T* x = static_cast<const T*>(X);
  const T* gg = static_cast<const T*>(g);
  T* y = static_cast<T*>(Y);
  const bool greg = static_cast<int>(grid.x) <= num_sms();
#define SF_RN(MV)                                                                                         \
  (greg ? launch_k(rmsnorm_rows_kernel<T, MV, true>, dim3(grid), dim3(block), 0, st, x, idx, n_dev, R, d,  \
                   gg, eps, y)                                                                           \
        : launch_k(rmsnorm_rows_kernel<T, MV, false>, dim3(grid), dim3(block), 0, st, x, idx, n_dev, R, d, \
                   gg, eps, y))
  if (per_lane <= 4)
    SF_RN(4);
  else if (per_lane <= 8)
    SF_RN(8);
  else if (per_lane <= 16)
    SF_RN(16);
  else
    SF_RN(32);
#undef SF_RN
}

int launch_rmsnorm_rows(int dtype, const void* X, const int32_t* idx, const int32_t* n_dev,
                        int R, int d, const void* g, float eps, void* Y, cudaStream_t st) {
  const int per_lane = (d / (dtype == SPECFOLD_BF16 ? 8 : 4) + 31) / 32;
  if (per_lane > 32) return SPECFOLD_EUNSUPPORTED;
  if (dtype == SPECFOLD_BF16)
    rmsnorm_dispatch<__nv_bfloat16>(X, idx, n_dev, R, d, g, eps, Y, st);
  else
    rmsnorm_dispatch<float>(X, idx, n_dev, R, d, g, eps, Y, st);
  count_launch();
  return check_launch();
}

int launch_fold_fill(int dtype, const uint8_t* fold, const int32_t* src, const void* H_in,
                     void* H_out, int R, int d, cudaStream_t st) {
  const dim3 grid((R + kRowWarps - 1) / kRowWarps), block(kRowWarps * 32);
  if (dtype == SPECFOLD_BF16)
    launch_k(fold_fill_kernel<__nv_bfloat16>, dim3(grid), dim3(block), 0, st, 
        fold, src, static_cast<const __nv_bfloat16*>(H_in), static_cast<__nv_bfloat16*>(H_out), R,
        d);
  else
    launch_k(fold_fill_kernel<float>, dim3(grid), dim3(block), 0, st, fold, src, static_cast<const float*>(H_in),
                                                    static_cast<float*>(H_out), R, d);
  count_launch();
  return check_launch();
}

int launch_gather_query(int dtype, const void* Q, const int32_t* src, const int32_t* slot, int R, int n_kv, int ghd,
                        void* Qall, int32_t* all_idx, int32_t* n_all, cudaStream_t st) {
  if ((ghd * (dtype == SPECFOLD_BF16 ? 2 : 4)) % 16) return SPECFOLD_EUNSUPPORTED;
  const dim3 grid((R * n_kv + kRowWarps - 1) / kRowWarps), block(kRowWarps * 32);
  if (dtype == SPECFOLD_BF16)
    launch_k(gather_query_kernel<__nv_bfloat16>, grid, block, 0, st, static_cast<const __nv_bfloat16*>(Q), src, slot,
             R, n_kv, ghd, static_cast<__nv_bfloat16*>(Qall), all_idx, n_all);
  else
    launch_k(gather_query_kernel<float>, grid, block, 0, st, static_cast<const float*>(Q), src, slot, R, n_kv, ghd,
             static_cast<float*>(Qall), all_idx, n_all);
  count_launch();
  return check_launch();
}

int launch_unpack_fill(int dtype, const void* Ap, const int32_t* src, const int32_t* slot, const void* H, void* Aall,
                       int R, int d, cudaStream_t st) {
  const dim3 grid((R + kRowWarps - 1) / kRowWarps), block(kRowWarps * 32);
  if (dtype == SPECFOLD_BF16)
    launch_k(unpack_fill_kernel<__nv_bfloat16>, grid, block, 0, st, static_cast<const __nv_bfloat16*>(Ap), src, slot,
             static_cast<const __nv_bfloat16*>(H), static_cast<__nv_bfloat16*>(Aall), R, d);
  else
    launch_k(unpack_fill_kernel<float>, grid, block, 0, st, static_cast<const float*>(Ap), src, slot,
             static_cast<const float*>(H), static_cast<float*>(Aall), R, d);
  count_launch();
  return check_launch();
}

int launch_timeout_probe(uint32_t* status, uint64_t wait_ns, cudaStream_t st) {
  timeout_probe_kernel<<<1, 32, 0, st>>>(status, wait_ns);
  count_launch();
  return check_launch();
}

}  // namespace sf
