// Persistent tcgen05 GEMM for the packed projections of the folded layer
// (QKV, output projection, SwiGLU gate/up, down projection).
//
//   D[k, c] = sum_j A[k, j] * W[c, j]      A: packed rows [Mcap, K] (bf16)
//                                          W: weights [N, K] (bf16, nn.Linear layout)
//
// One CTA per SM loops over work units (m-tile, k-split, n-tile).  The number
// of packed rows n is read on the device, so the decomposition adapts to the
// recompute fraction without a host round trip: when the m x n tiles cannot
// fill the SMs, the K loop is split across CTAs.  Two ways to sum the splits:
//   * clustered launch (when the host knows every n leaves SMs idle): the S
//     CTAs of one tile sit in one thread-block cluster; each stages its fp32
//     partial tile in its own shared memory, and after a cluster barrier each
//     sums a 1/S column share of the tile from all S stages through
//     distributed shared memory, in split order, and runs the epilogue;
//   * otherwise each CTA writes its fp32 partial tile to global memory and a
//     second, fully parallel kernel sums them in split order.
// Both orders are fixed, so results are deterministic.
//
// Roles (192 threads): warp 0 issues TMA loads into a multi-stage ring of
// 128-byte-swizzled tiles; warp 1 allocates TMEM and issues tcgen05.mma
// (M = 128, N = BN, K = 16 per instruction) into one of two TMEM accumulators;
// warps 2-5 read the accumulator back with tcgen05.ld (one row per thread)
// and run the fused epilogue while the next unit accumulates.
#include "sf_device.cuh"
#include "sf_internal.h"

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace sf {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;              // 128 bytes of bf16: one swizzle atom row
constexpr int kGemmThreads = 192;
constexpr int kMaxGrid = 160;        // persistent CTAs (>= SMs of one GB300)
constexpr int kMaxSplits = 16;
constexpr int kMinKbPerSplit = 4;
constexpr int kMaxClusterSplit = 8;  // largest cluster (portable size)
constexpr int kSchedRows = SPECFOLD_MAX_ROWS / 128;  // m-tile counts

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_BYTES = 256;
  static constexpr int EPI_STAGE_BYTES = 4 * 32 * 33 * 4;  // per epilogue warp: 32 x 32 fp32, padded
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + EPI_STAGE_BYTES + 1024;
  // clustered split: the fp32 partial tile, rows padded by 16 bytes, staged
  // over the operand ring once the CTA's only unit has consumed it
  static constexpr int SROW = BN + 4;
  static_assert(kBM * SROW * 4 + kBM * 4 <= STAGES * STAGE_BYTES, "partial tile and row indices must fit the ring");
};

struct GemmParams {
  CUtensorMap mapA;
  CUtensorMap mapB[3];
  int col0[3];          // first output column of each stacked weight
  int nb;
  int K, Mcap, N, Nt;
  const int32_t* n_dev;
  void* Y;
  long long ldy;
  const void* resid;
  long long ldr;
  const int32_t* row_idx;
  void* Yk;
  void* Yv;
  int n_q, n_kv, hd, g, R;
  float* partial;
  uint32_t* status;
  int cs;               // cluster size of a clustered launch (0: plain launch)
  const int32_t* dep_rng;   // RESID_SCATTER: fold-fill of dependents in the finish kernel
  const int32_t* dep_rows;
  const __nv_bfloat16* hin;
  const int32_t* fill_src;  // RESID_SCATTER: the two-pass finish (fold-fill by folded row, from src)
  uint32_t* fill_bar;       // its grid-barrier word
  int n_early;              // n_dev and row_idx may be read before the programmatic wait
  // work decomposition per m-tile count Mt (row Mt - 1): S, full, r, St, U
  // (see Sched); filled by the host for this launch's grid
  int sched[kSchedRows][5];
};

SF_DEV float silu(float x) { return __fdividef(x, 1.f + ex2(-x * 1.4426950408889634f)); }

template <int W>
SF_DEV void store_bf16(__nv_bfloat16* dst, const float (&v)[W]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < W / 8; ++q)
    d4[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                       pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}
template <int W>
SF_DEV void add_bf16(const __nv_bfloat16* src, float (&v)[W]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < W / 8; ++q) {
    const uint4 u = __ldg(s4 + q);
    v[8 * q + 0] += bf16lo(u.x); v[8 * q + 1] += bf16hi(u.x);
    v[8 * q + 2] += bf16lo(u.y); v[8 * q + 3] += bf16hi(u.y);
    v[8 * q + 4] += bf16lo(u.z); v[8 * q + 5] += bf16hi(u.z);
    v[8 * q + 6] += bf16lo(u.w); v[8 * q + 7] += bf16hi(u.w);
  }
}

// Epilogue of W consecutive output columns of packed row k.  c = first output
// column (first feature for SWIGLU, where v holds gate and u holds up values).
template <int EPI, int W>
SF_DEV void epi_chunk(const GemmParams& p, int k, int c, float (&v)[W], const float (&u)[W]) {
  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(p.Y);
  if constexpr (EPI == EPI_STORE) {
    store_bf16<W>(Y + static_cast<size_t>(k) * p.ldy + c, v);
  } else if constexpr (EPI == EPI_RESID_PACKED) {
    const int r = p.row_idx[k];
    add_bf16<W>(static_cast<const __nv_bfloat16*>(p.resid) + static_cast<size_t>(r) * p.ldr + c, v);
    store_bf16<W>(Y + static_cast<size_t>(k) * p.ldy + c, v);
  } else if constexpr (EPI == EPI_RESID_SCATTER) {
    const int r = p.row_idx[k];
    add_bf16<W>(static_cast<const __nv_bfloat16*>(p.resid) + static_cast<size_t>(k) * p.ldr + c, v);
    store_bf16<W>(Y + static_cast<size_t>(r) * p.ldy + c, v);
  } else if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll
    for (int e = 0; e < W; ++e) v[e] = silu(v[e]) * u[e];
    store_bf16<W>(Y + static_cast<size_t>(k) * p.ldy + c, v);
  } else {  // EPI_QKV: W columns never straddle a head (hd % 32 == 0)
    const int nq = p.n_q * p.hd, nkv = p.n_kv * p.hd;
    if (c < nq) {
      const int head = c / p.hd, j = c - head * p.hd;
      const int hk = head / p.g, hg = head - hk * p.g;
      store_bf16<W>(Y + ((static_cast<size_t>(hk) * p.R + k) * p.g + hg) * p.hd + j, v);
    } else {
      const int r = p.row_idx[k];
      const bool is_k = c < nq + nkv;
      const int cc = is_k ? c - nq : c - nq - nkv;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(is_k ? p.Yk : p.Yv);
      store_bf16<W>(dst + static_cast<size_t>(r) * nkv + cc, v);
    }
  }
}

// Split factor of the K loop for n packed rows: only when the m x n tiles
// cannot fill the grid, and never below kMinKbPerSplit k-blocks per split.
__host__ __device__ inline int split_factor(int tiles, int grid, int KB) {
  int S = 1;
  if (tiles > 0 && tiles < grid) {
    S = grid / tiles < KB / kMinKbPerSplit ? grid / tiles : KB / kMinKbPerSplit;
    S = S < kMaxSplits ? S : kMaxSplits;
    S = S > 1 ? S : 1;
  }
  return S;
}

// Epilogue of one output element (row k, column c); for SWIGLU x is the
// gate value and u the up value of feature c.
template <int EPI>
SF_DEV void epi_elem(const GemmParams& p, int k, int c, float x, float u) {
  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(p.Y);
  const __nv_bfloat16* Rz = static_cast<const __nv_bfloat16*>(p.resid);
  if constexpr (EPI == EPI_STORE) {
    Y[static_cast<size_t>(k) * p.ldy + c] = __float2bfloat16_rn(x);
  } else if constexpr (EPI == EPI_RESID_PACKED) {
    const int r = p.row_idx[k];
    Y[static_cast<size_t>(k) * p.ldy + c] = __float2bfloat16_rn(x + __bfloat162float(Rz[static_cast<size_t>(r) * p.ldr + c]));
  } else if constexpr (EPI == EPI_RESID_SCATTER) {
    const int r = p.row_idx[k];
    Y[static_cast<size_t>(r) * p.ldy + c] = __float2bfloat16_rn(x + __bfloat162float(Rz[static_cast<size_t>(k) * p.ldr + c]));
  } else if constexpr (EPI == EPI_SWIGLU) {
    Y[static_cast<size_t>(k) * p.ldy + c] = __float2bfloat16_rn(silu(x) * u);
  } else {  // EPI_QKV
    const int nq = p.n_q * p.hd, nkv = p.n_kv * p.hd;
    if (c < nq) {
      const int head = c / p.hd, j = c - head * p.hd;
      const int hk = head / p.g, hg = head - hk * p.g;
      Y[((static_cast<size_t>(hk) * p.R + k) * p.g + hg) * p.hd + j] = __float2bfloat16_rn(x);
    } else {
      const int r = p.row_idx[k];
      const bool is_k = c < nq + nkv;
      const int cc = is_k ? c - nq : c - nq - nkv;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(is_k ? p.Yk : p.Yv);
      dst[static_cast<size_t>(r) * nkv + cc] = __float2bfloat16_rn(x);
    }
  }
}

// Split factor under clusters of cs CTAs: the largest divisor of cs that keeps
// tiles * S within the grid and kMinKbPerSplit k-blocks per split.
SF_DEV int split_factor_cl(int tiles, int grid, int KB, int cs) {
  for (int S = cs; S > 1; --S)
    if (cs % S == 0 && tiles * S <= grid && KB / S >= kMinKbPerSplit) return S;
  return 1;
}

struct Unit {
  int m, s, nt, kb0, kb1, tile;
  int slot;    // fp32 partial tile written by a split unit
  bool split;  // the unit covers part of its tile's K range
};

// Work decomposition of a plain launch for n packed rows on G CTAs.  When
// the tiles cannot fill the grid, every tile's K loop is split S ways.  When
// they can, the last partial wave would leave SMs idle: if it holds at most
// half a wave (r tiles), those r tiles are split St ways instead, so the
// last wave is full and each of its units is St times shorter.
struct Sched {
  int Mt, tiles, KB;
  int S;         // split of every tile (tiles < G), else 1
  int full;      // units [0, full) are whole tiles
  int r, St;     // the last r tiles split St ways (St >= 2), else r = 0, St = 1
  int U;         // units
};

__host__ __device__ inline Sched make_sched(int n, int Nt, int G, int KB) {
  Sched c;
  c.Mt = (n + kBM - 1) / kBM;
  c.tiles = c.Mt * Nt;
  c.KB = KB;
  c.S = 1;
  c.full = c.tiles;
  c.r = 0;
  c.St = 1;
  if (c.tiles < G) {
    c.S = split_factor(c.tiles, G, KB);
  } else {
    const int r = c.tiles % G;
    if (r > 0 && 2 * r <= G) {
      int St = G / r < KB / kMinKbPerSplit ? G / r : KB / kMinKbPerSplit;
      St = St < kMaxSplits ? St : kMaxSplits;
      if (St >= 2) {
        c.r = r;
        c.St = St;
        c.full = c.tiles - r;
      }
    }
  }
  c.U = c.S > 1 ? c.tiles * c.S : c.full + c.r * c.St;
  return c;
}

// The launch's schedule for n rows, from the host-filled table.
SF_DEV Sched get_sched(const int (&tab)[kSchedRows][5], int n, int Nt, int KB) {
  Sched c;
  c.Mt = (n + kBM - 1) / kBM;
  c.tiles = c.Mt * Nt;
  c.KB = KB;
  if (c.Mt <= 0 || c.Mt > kSchedRows) {
    c.S = 1, c.full = c.tiles, c.r = 0, c.St = 1, c.U = c.tiles;
    return c;
  }
  const int* e = tab[c.Mt - 1];
  c.S = e[0], c.full = e[1], c.r = e[2], c.St = e[3], c.U = e[4];
  return c;
}

SF_DEV Unit decode_plain(int u, const Sched& c, int Nt) {
  Unit w;
  if (c.S > 1) {
    w.m = u % c.Mt;
    const int rest = u / c.Mt;
    w.s = rest % c.S;
    w.nt = rest / c.S;
    w.kb0 = (w.s * c.KB) / c.S;
    w.kb1 = ((w.s + 1) * c.KB) / c.S;
    w.tile = w.m * Nt + w.nt;
    w.slot = w.tile * c.S + w.s;
    w.split = true;
  } else if (u < c.full) {
    w.m = u % c.Mt;
    w.nt = u / c.Mt;
    w.s = 0;
    w.kb0 = 0;
    w.kb1 = c.KB;
    w.tile = w.m * Nt + w.nt;
    w.slot = 0;
    w.split = false;
  } else {
    const int v = u - c.full;
    const int q = v / c.St;
    w.s = v - q * c.St;
    const int t = c.full + q;  // whole-tile unit index of this tail tile
    w.m = t % c.Mt;
    w.nt = t / c.Mt;
    w.kb0 = (w.s * c.KB) / c.St;
    w.kb1 = ((w.s + 1) * c.KB) / c.St;
    w.tile = w.m * Nt + w.nt;
    w.slot = q * c.St + w.s;
    w.split = true;
  }
  return w;
}

// Whether tile (m, nt) was split, by how many, and its first partial slot.
SF_DEV bool tile_split(const Sched& c, int m, int nt, int Nt, int& nsplit, int& slot0) {
  if (c.S > 1) {
    nsplit = c.S;
    slot0 = (m * Nt + nt) * c.S;
    return true;
  }
  if (c.St > 1) {
    const int u = m + c.Mt * nt;
    if (u >= c.full) {
      nsplit = c.St;
      slot0 = (u - c.full) * c.St;
      return true;
    }
  }
  return false;
}

// Work unit u.  Plain: m fastest, then split, then n-tile.  Clustered split
// (dsm): the S consecutive CTAs u = tile * S + s share one tile, so they sit
// in one cluster (S divides the cluster size).
SF_DEV Unit decode(int u, int Mt, int S, int Nt, int KB, bool dsm) {
  Unit w;
  if (dsm) {
    w.s = u % S;
    const int tile = u / S;
    w.m = tile % Mt;
    w.nt = tile / Mt;
  } else {
    w.m = u % Mt;
    const int rest = u / Mt;
    w.s = rest % S;
    w.nt = rest / S;
  }
  w.kb0 = (w.s * KB) / S;
  w.kb1 = ((w.s + 1) * KB) / S;
  w.tile = w.m * Nt + w.nt;
  w.slot = w.tile * S + w.s;
  w.split = S > 1;
  return w;
}

// Clustered split-K finish: this CTA (split s of its tile) sums output
// columns [s, s + 1) * TW / S of every valid row over the S partial tiles
// staged in the group's shared memories, in split order, and runs the
// epilogue on groups of 8 columns.  The row indices were staged next to the
// partial tile, so every global load of an item (residual row) is issued
// before its distributed-shared-memory loads and the two latencies overlap.
// SC is the split count; a thread issues the loads of ITEMS items (2·SC
// distributed-shared-memory vectors each, 16 in all) before it sums any of
// them, so their latencies overlap too.
template <int BN, int EPI, int SC>
SF_DEV void dsm_reduce_sc(const GemmParams& p, const uint8_t* smem, int n, int Mt) {
  constexpr int TW = EPI == EPI_SWIGLU ? BN / 2 : BN;  // output columns per tile
  constexpr int SROW = Cfg<BN>::SROW;
  constexpr int HALVES = EPI == EPI_SWIGLU ? 2 : 1;    // gate and up columns
  constexpr int ITEMS = (8 / SC) / HALVES > 0 ? (8 / SC) / HALVES : 1;
  const int* s_ridx = reinterpret_cast<const int*>(smem + kBM * SROW * 4);
  const int s = static_cast<int>(blockIdx.x) % SC;
  const uint32_t rank0 = cluster_ctarank() - static_cast<uint32_t>(s);
  const int tile = static_cast<int>(blockIdx.x) / SC;
  const int m = tile % Mt, nt = tile / Mt;
  const int rows = min(kBM, n - m * kBM);
  constexpr int share = TW / SC;
  constexpr int groups = share / 8;
  const uint32_t sbase = smem_u32(smem);
  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(p.Y);
  const __nv_bfloat16* Rz = static_cast<const __nv_bfloat16*>(p.resid);
  const int total = rows * groups;
  for (int idx0 = threadIdx.x; idx0 < total; idx0 += ITEMS * kGemmThreads) {
    float4 a[ITEMS][SC][2], b[ITEMS][SC][2];
    uint4 res[ITEMS];
    // every load of the thread's items first
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int idx = idx0 + it * kGemmThreads;
      if (idx >= total) break;
      const int r = idx / groups;
      const int tc = s * share + (idx - r * groups) * 8;
      const int k = m * kBM + r;
      const int c = nt * TW + tc;
      res[it] = make_uint4(0, 0, 0, 0);
      if constexpr (EPI == EPI_RESID_PACKED)
        res[it] = __ldg(reinterpret_cast<const uint4*>(Rz + static_cast<size_t>(s_ridx[r]) * p.ldr + c));
      if constexpr (EPI == EPI_RESID_SCATTER)
        res[it] = __ldg(reinterpret_cast<const uint4*>(Rz + static_cast<size_t>(k) * p.ldr + c));
      const uint32_t off = sbase + static_cast<uint32_t>((r * SROW + tc) * 4);
#pragma unroll
      for (int j = 0; j < SC; ++j) {
        const uint32_t ra = dsmem_addr(off, rank0 + j);
        a[it][j][0] = ld_dsmem_f4(ra);
        a[it][j][1] = ld_dsmem_f4(ra + 16);
        if constexpr (EPI == EPI_SWIGLU) {
          b[it][j][0] = ld_dsmem_f4(ra + (BN / 2) * 4);
          b[it][j][1] = ld_dsmem_f4(ra + (BN / 2) * 4 + 16);
        }
      }
    }
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int idx = idx0 + it * kGemmThreads;
      if (idx >= total) break;
      const int r = idx / groups;
      const int tc = s * share + (idx - r * groups) * 8;
      const int k = m * kBM + r;
      const int c = nt * TW + tc;
      float v[8], u[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = u[e] = 0.f;
#pragma unroll
      for (int j = 0; j < SC; ++j) {
        v[0] += a[it][j][0].x; v[1] += a[it][j][0].y; v[2] += a[it][j][0].z; v[3] += a[it][j][0].w;
        v[4] += a[it][j][1].x; v[5] += a[it][j][1].y; v[6] += a[it][j][1].z; v[7] += a[it][j][1].w;
        if constexpr (EPI == EPI_SWIGLU) {
          u[0] += b[it][j][0].x; u[1] += b[it][j][0].y; u[2] += b[it][j][0].z; u[3] += b[it][j][0].w;
          u[4] += b[it][j][1].x; u[5] += b[it][j][1].y; u[6] += b[it][j][1].z; u[7] += b[it][j][1].w;
        }
      }
      if constexpr (EPI == EPI_RESID_PACKED || EPI == EPI_RESID_SCATTER) {
        const uint4 rs = res[it];
        v[0] += bf16lo(rs.x); v[1] += bf16hi(rs.x); v[2] += bf16lo(rs.y); v[3] += bf16hi(rs.y);
        v[4] += bf16lo(rs.z); v[5] += bf16hi(rs.z); v[6] += bf16lo(rs.w); v[7] += bf16hi(rs.w);
        const int rdst = EPI == EPI_RESID_PACKED ? k : s_ridx[r];
        store_bf16<8>(Y + static_cast<size_t>(rdst) * p.ldy + c, v);
      } else if constexpr (EPI == EPI_QKV) {
        const int nq = p.n_q * p.hd, nkv = p.n_kv * p.hd;
        if (c < nq) {
          const int head = c / p.hd, jh = c - head * p.hd;
          const int hk = head / p.g, hg = head - hk * p.g;
          store_bf16<8>(Y + ((static_cast<size_t>(hk) * p.R + k) * p.g + hg) * p.hd + jh, v);
        } else {
          const bool is_k = c < nq + nkv;
          const int cc = is_k ? c - nq : c - nq - nkv;
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(is_k ? p.Yk : p.Yv);
          store_bf16<8>(dst + static_cast<size_t>(s_ridx[r]) * nkv + cc, v);
        }
      } else {
        epi_chunk<EPI, 8>(p, k, c, v, u);
      }
    }
  }
}

// The split count of a clustered launch divides the cluster size (2, 4 or 8).
template <int BN, int EPI>
SF_DEV void dsm_reduce(const GemmParams& p, const uint8_t* smem, int n, int Mt, int S) {
  if (S == 2) dsm_reduce_sc<BN, EPI, 2>(p, smem, n, Mt);
  else if (S == 4) dsm_reduce_sc<BN, EPI, 4>(p, smem, n, Mt);
  else if (S == 8) dsm_reduce_sc<BN, EPI, 8>(p, smem, n, Mt);
}

template <int BN, int EPI, bool CL>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, kept in the shared state space (see attn_tc.cu)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* accf = bars + 2 * C::STAGES;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = abort_flag + 1;    // accumulator-ready broadcast
  float* epi_stage = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES + C::BAR_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // n through L2, early, when its producer is known complete (n_early)
  const int n_pre = p.n_early && p.n_dev ? __ldcg(p.n_dev) : 0;
  // Set-up that depends on no earlier kernel runs before the programmatic
  // wait, overlapping the previous kernel's tail wherever this CTA is already
  // resident: barriers, tensor-map prefetch, TMEM.  (A GEMM CTA shares an SM
  // only with kernels that hold no TMEM -- the row and finish kernels --
  // since attention and the other GEMMs take too much shared memory to fit
  // beside it, so the allocation cannot wait on a kernel that waits on it.)
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&accf[i]), 1);
      mbar_init(smem_u32(&acce[i]), 128);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.mapA);
    for (int j = 0; j < p.nb; ++j) prefetch_tmap(&p.mapB[j]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The FFN GEMMs' weight tiles: the first unit's first kPreB stages of B go
  // out before the wait when n is known early (the weights are an input; A,
  // the previous kernel's output, follows after the wait on the same
  // barriers).  Their predecessors (the output-projection finish, the gate/up
  // GEMM's tail) leave DRAM time to spare.
  constexpr int kPreB = 4;
  int preb = 0;
  auto b_coords = [&](const Unit& w, const CUtensorMap*& mlo, const CUtensorMap*& mhi, int& ylo, int& yhi) {
    if constexpr (EPI == EPI_SWIGLU) {
      mlo = &p.mapB[0];
      mhi = &p.mapB[1];
      ylo = yhi = w.nt * (BN / 2);
    } else {
      const int c0 = w.nt * BN;
      int j = 0;
      while (j + 1 < p.nb && c0 >= p.col0[j + 1]) ++j;
      mlo = mhi = &p.mapB[j];
      ylo = c0 - p.col0[j];
      yhi = ylo + BN / 2;
    }
  };
  if constexpr (!CL && (EPI == EPI_SWIGLU || EPI == EPI_RESID_SCATTER)) {
    if (p.n_early && warp == 0 && lane == 0) {
      const int n0 = p.n_dev ? min(max(n_pre, 0), p.Mcap) : p.Mcap;
      const Sched sc0 = get_sched(p.sched, n0, p.Nt, p.K / kBK);
      if (static_cast<int>(blockIdx.x) < sc0.U) {
        const Unit w = decode_plain(static_cast<int>(blockIdx.x), sc0, p.Nt);
        const CUtensorMap* mlo;
        const CUtensorMap* mhi;
        int ylo, yhi;
        b_coords(w, mlo, mhi, ylo, yhi);
        preb = min(min(kPreB, C::STAGES), w.kb1 - w.kb0);
        for (int it = 0; it < preb; ++it) {  // fresh stages: nothing to wait for
          uint8_t* sb = smem + it * C::STAGE_BYTES + C::A_BYTES;
          const uint32_t fb = smem_u32(&full[it]);
          mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          tma_load_2d(smem_u32(sb), mlo, fb, (w.kb0 + it) * kBK, ylo);
          tma_load_2d(smem_u32(sb + (BN / 2) * 128), mhi, fb, (w.kb0 + it) * kBK, yhi);
        }
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  const int n = p.n_dev ? min(max(p.n_early ? n_pre : p.n_dev[0], 0), p.Mcap) : p.Mcap;
  const int Mt = (n + kBM - 1) / kBM;
  const int tiles = Mt * p.Nt;
  const int KB = p.K / kBK;
  const Sched sc = get_sched(p.sched, n, p.Nt, KB);
  const int S = CL ? split_factor_cl(tiles, static_cast<int>(gridDim.x), KB, p.cs) : sc.S;
  const bool dsm = CL && S > 1;  // splits summed through distributed shared memory
  const int U = CL ? tiles * S : sc.U;
  auto unit = [&](int u) { return CL ? decode(u, Mt, S, p.Nt, KB, dsm) : decode_plain(u, sc, p.Nt); };
  if (static_cast<int>(blockIdx.x) >= U) {
    if (warp == 1) tmem_dealloc(*tmem_slot, C::TMEM_COLS);
    if constexpr (CL) {
      if (dsm) {  // an idle CTA still takes part in its cluster's two barriers
        cluster_sync_all();
        cluster_sync_all();
      }
    }
    return;
  }

  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
        const Unit w = unit(u);
        const CUtensorMap* mlo;
        const CUtensorMap* mhi;
        int ylo, yhi;
        b_coords(w, mlo, mhi, ylo, yhi);
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int st = it % C::STAGES;
          uint8_t* sa = smem + st * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          const uint32_t fb = smem_u32(&full[st]);
          if (static_cast<int>(it) < preb) {  // B already on its way (before the wait)
            tma_load_2d(smem_u32(sa), &p.mapA, fb, kb * kBK, w.m * kBM);
            continue;
          }
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1, abort_flag, p.status, kWaitLimitNs, kSiteGemmEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          tma_load_2d(smem_u32(sa), &p.mapA, fb, kb * kBK, w.m * kBM);
          tma_load_2d(smem_u32(sb), mlo, fb, kb * kBK, ylo);
          tma_load_2d(smem_u32(sb + (BN / 2) * 128), mhi, fb, kb * kBK, yhi);
        }
      }
      if (!ok && it > 0) {
        // let the loads already issued land before the CTA exits
        int never = 0;
        const uint32_t last = it - 1;
        mbar_wait(smem_u32(&full[last % C::STAGES]), (last / C::STAGES) & 1, &never, nullptr,
                  10000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, false);
      uint32_t it = 0, t = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++t) {
        const Unit w = unit(u);
        const int ab = t & 1;
        if (!mbar_wait(smem_u32(&acce[ab]), ((t >> 1) & 1) ^ 1, abort_flag, p.status, kWaitLimitNs, kSiteGemmAccEmpty)) break;
        tc_fence_after();
        const uint32_t dt = tmem_base + ab * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(smem_u32(&full[st]), ph, abort_flag, p.status, kWaitLimitNs, kSiteGemmFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + st * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            tc_mma_f16(dt, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024),
                       idesc, (kb > w.kb0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(smem_u32(&empty[st]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&accf[ab]));
      }
      // every MMA issued must complete before TMEM is released
      tc_commit(smem_u32(drain));
      int never = 0;
      mbar_wait(smem_u32(drain), 0, &never, nullptr, 10000000ull);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue --
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int et = threadIdx.x - 64;    // 0..127
    uint32_t t = 0;
    for (int u = blockIdx.x; u < U; u += gridDim.x, ++t) {
      const Unit w = unit(u);
      const int ab = t & 1;
      if (et == 0) *s_ok = mbar_wait(smem_u32(&accf[ab]), (t >> 1) & 1, abort_flag, p.status, kWaitLimitNs, kSiteGemmAccFull) ? 1 : 0;
      named_bar_sync(1, 128);
      const bool ok = *s_ok != 0;
      named_bar_sync(1, 128);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * BN;
      if (dsm) {
        // this CTA's only unit: stage its fp32 partial tile (one row per
        // thread) over the operand ring, whose loads have all been consumed
        float* dst = reinterpret_cast<float*>(smem) + (q * 32 + lane) * C::SROW;
        if constexpr (EPI == EPI_QKV || EPI == EPI_RESID_PACKED || EPI == EPI_RESID_SCATTER) {
          const int row = w.m * kBM + q * 32 + lane;
          reinterpret_cast<int*>(smem + kBM * C::SROW * 4)[q * 32 + lane] = row < n ? p.row_idx[row] : 0;
        }
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(tb + ch * 32, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4)
            reinterpret_cast<float4*>(dst + ch * 32)[e4] =
                make_float4(__uint_as_float(r[4 * e4]), __uint_as_float(r[4 * e4 + 1]),
                            __uint_as_float(r[4 * e4 + 2]), __uint_as_float(r[4 * e4 + 3]));
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&acce[ab]));
        continue;
      }
      const int row0 = w.m * kBM + q * 32;          // first packed row of this warp
      const int rows_here = min(32, n - row0);      // valid rows (may be <= 0)
      if constexpr (EPI == EPI_QKV) {
        if (!w.split) {
          // straight from TMEM as for SwiGLU below: thread `lane` owns row
          // row0 + lane; a 32-column chunk lies in one head (hd % 32 == 0), so
          // its 32 values go out as 64 contiguous bytes, to the head-group
          // major Q or to the K/V row of the packed row's source row
          const int k = row0 + lane;
          const bool valid = lane < rows_here;
          const int ridx_row = valid ? p.row_idx[k] : 0;
          const int nq = p.n_q * p.hd, nkv = p.n_kv * p.hd;
          __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(p.Y);
#pragma unroll 1
          for (int ch = 0; ch < BN / 32; ++ch) {
            uint32_t r[32];
            tmem_ld32(tb + ch * 32, r);
            tmem_ld_wait(r);
            if (valid) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 32; e += 2) pk[e / 2] = pack_bf16x2(__uint_as_float(r[e]), __uint_as_float(r[e + 1]));
              const int cbase = w.nt * BN + ch * 32;
              __nv_bfloat16* dst;
              if (cbase < nq) {
                const int head = cbase / p.hd;
                const int hk = head / p.g, hg = head - hk * p.g;
                dst = Y + ((static_cast<size_t>(hk) * p.R + k) * p.g + hg) * p.hd + (cbase - head * p.hd);
              } else {
                const bool is_k = cbase < nq + nkv;
                dst = static_cast<__nv_bfloat16*>(is_k ? p.Yk : p.Yv) + static_cast<size_t>(ridx_row) * nkv +
                      (is_k ? cbase - nq : cbase - nq - nkv);
              }
              uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) d4[q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
            }
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&acce[ab]));
          continue;
        }
      }
      if constexpr (EPI == EPI_RESID_PACKED || EPI == EPI_RESID_SCATTER) {
        if (!w.split) {
          // straight from TMEM as for QKV above: thread `lane` owns row
          // row0 + lane, adds its residual row's chunk (64 contiguous bytes,
          // two chunks' loads in flight) and writes 64 contiguous bytes --
          // packed row k (output projection) or row row_idx[k] (down)
          const int k = row0 + lane;
          const bool valid = lane < rows_here;
          const int ridx_row = valid ? p.row_idx[k] : 0;
          const int rres = EPI == EPI_RESID_PACKED ? ridx_row : k;   // residual row
          const int rdst = EPI == EPI_RESID_PACKED ? k : ridx_row;   // output row
          const __nv_bfloat16* Rz = static_cast<const __nv_bfloat16*>(p.resid) + static_cast<size_t>(rres) * p.ldr;
          __nv_bfloat16* Yr = static_cast<__nv_bfloat16*>(p.Y) + static_cast<size_t>(rdst) * p.ldy;
#pragma unroll 1
          for (int ch = 0; ch < BN / 32; ch += 2) {
            uint4 rv[2][4];
            if (valid) {
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                  rv[h2][q4] = __ldg(reinterpret_cast<const uint4*>(Rz + w.nt * BN + (ch + h2) * 32) + q4);
            }
            uint32_t r0[32], r1[32];
            tmem_ld32(tb + ch * 32, r0);
            tmem_ld32(tb + (ch + 1) * 32, r1);
            tmem_ld_wait(r0);
            tmem_ld_wait(r1);
            if (valid) {
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t* rr = h2 ? r1 : r0;
                uint4* d4 = reinterpret_cast<uint4*>(Yr + w.nt * BN + (ch + h2) * 32);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const uint4 u = rv[h2][q4];
                  const int e0 = q4 * 8;
                  d4[q4] = make_uint4(
                      pack_bf16x2(__uint_as_float(rr[e0 + 0]) + bf16lo(u.x), __uint_as_float(rr[e0 + 1]) + bf16hi(u.x)),
                      pack_bf16x2(__uint_as_float(rr[e0 + 2]) + bf16lo(u.y), __uint_as_float(rr[e0 + 3]) + bf16hi(u.y)),
                      pack_bf16x2(__uint_as_float(rr[e0 + 4]) + bf16lo(u.z), __uint_as_float(rr[e0 + 5]) + bf16hi(u.z)),
                      pack_bf16x2(__uint_as_float(rr[e0 + 6]) + bf16lo(u.w), __uint_as_float(rr[e0 + 7]) + bf16hi(u.w)));
                }
              }
            }
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&acce[ab]));
          continue;
        }
      }
      if constexpr (EPI == EPI_SWIGLU || EPI == EPI_STORE) {
        if (!w.split) {
          // Straight from TMEM: thread `lane` owns row row0 + lane and writes
          // each 32-column chunk of it as 64 contiguous bytes (four 16-byte
          // stores), with no shared-memory transpose and no per-element
          // branch (the transposed path's dependent chains left the last
          // tile's SwiGLU epilogue exposed for several microseconds)
          __nv_bfloat16* yrow = static_cast<__nv_bfloat16*>(p.Y) + static_cast<size_t>(row0 + lane) * p.ldy;
          constexpr int NCH = EPI == EPI_SWIGLU ? BN / 64 : BN / 32;
#pragma unroll 1
          for (int ch = 0; ch < NCH; ++ch) {
            uint32_t r[32];
            tmem_ld32(tb + ch * 32, r);
            uint32_t pk[16];
            if constexpr (EPI == EPI_SWIGLU) {
              uint32_t r2[32];
              tmem_ld32(tb + BN / 2 + ch * 32, r2);
              tmem_ld_wait(r);
              tmem_ld_wait(r2);
#pragma unroll
              for (int e = 0; e < 32; e += 2)
                pk[e / 2] = pack_bf16x2(silu(__uint_as_float(r[e])) * __uint_as_float(r2[e]),
                                        silu(__uint_as_float(r[e + 1])) * __uint_as_float(r2[e + 1]));
            } else {
              tmem_ld_wait(r);
#pragma unroll
              for (int e = 0; e < 32; e += 2) pk[e / 2] = pack_bf16x2(__uint_as_float(r[e]), __uint_as_float(r[e + 1]));
            }
            if (lane < rows_here) {
              const int c = (EPI == EPI_SWIGLU ? w.nt * (BN / 2) : w.nt * BN) + ch * 32;
              uint4* dst = reinterpret_cast<uint4*>(yrow + c);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) dst[q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
            }
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&acce[ab]));
          continue;
        }
      }
      // Each 32-column chunk of the warp's 32 rows goes through a padded smem
      // transpose so that lane j then handles column j of one row at a time:
      // every store (and residual load) of the warp is one contiguous segment.
      float* stg = epi_stage + q * (32 * 33);
      // lane j holds the row index of the warp's row j (broadcast by shuffle)
      int ridx = 0;
      if constexpr (EPI == EPI_QKV || EPI == EPI_RESID_PACKED || EPI == EPI_RESID_SCATTER)
        if (!w.split && lane < rows_here) ridx = p.row_idx[row0 + lane];
      float* prow = p.partial + static_cast<size_t>(w.slot) * kBM * BN + static_cast<size_t>(q * 32) * BN;
      constexpr int NCH = EPI == EPI_SWIGLU ? BN / 64 : BN / 32;
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t r[32];
        tmem_ld32(tb + ch * 32, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int e = 0; e < 32; ++e) stg[lane * 33 + e] = __uint_as_float(r[e]);
        float gt[32];  // SWIGLU: gate values of column `lane`, one per row
        if constexpr (EPI == EPI_SWIGLU) {
          // the up half of the tile: same rows, columns BN/2 further on
          uint32_t r2[32];
          tmem_ld32(tb + BN / 2 + ch * 32, r2);
          tmem_ld_wait(r2);
          __syncwarp();
#pragma unroll
          for (int rr = 0; rr < 32; ++rr) gt[rr] = stg[rr * 33 + lane];
          __syncwarp();
#pragma unroll
          for (int e = 0; e < 32; ++e) stg[lane * 33 + e] = __uint_as_float(r2[e]);
        }
        __syncwarp();
        if (!w.split) {
          const int cbase = EPI == EPI_SWIGLU ? w.nt * (BN / 2) + ch * 32 : w.nt * BN + ch * 32;
          const int c = cbase + lane;
          __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(p.Y);
          const __nv_bfloat16* Rz = static_cast<const __nv_bfloat16*>(p.resid);
          if constexpr (EPI == EPI_RESID_PACKED || EPI == EPI_RESID_SCATTER) {
            // all 32 residual loads of the chunk are in flight before any store
            float rv[32];
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
              const int rres = EPI == EPI_RESID_PACKED ? __shfl_sync(0xffffffffu, ridx, rr) : row0 + rr;
              rv[rr] = rr < rows_here ? __bfloat162float(Rz[static_cast<size_t>(rres) * p.ldr + c]) : 0.f;
            }
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
              const int rdst = EPI == EPI_RESID_PACKED ? row0 + rr : __shfl_sync(0xffffffffu, ridx, rr);
              if (rr < rows_here)
                Y[static_cast<size_t>(rdst) * p.ldy + c] = __float2bfloat16_rn(stg[rr * 33 + lane] + rv[rr]);
            }
          } else if constexpr (EPI == EPI_QKV) {
            // the 32 columns of a chunk lie in one head (hd % 32 == 0): the
            // destination is decomposed once per chunk, not per element
            const int nq = p.n_q * p.hd, nkv = p.n_kv * p.hd;
            if (cbase < nq) {
              const int head = cbase / p.hd;
              const int hk = head / p.g, hg = head - hk * p.g;
              const size_t rstride = static_cast<size_t>(p.g) * p.hd;
              __nv_bfloat16* qb = Y + (static_cast<size_t>(hk) * p.R * p.g + hg) * p.hd + (cbase - head * p.hd) + lane;
#pragma unroll
              for (int rr = 0; rr < 32; ++rr)
                if (rr < rows_here) qb[static_cast<size_t>(row0 + rr) * rstride] = __float2bfloat16_rn(stg[rr * 33 + lane]);
            } else {
              const bool is_k = cbase < nq + nkv;
              __nv_bfloat16* kb = static_cast<__nv_bfloat16*>(is_k ? p.Yk : p.Yv) +
                                  (is_k ? cbase - nq : cbase - nq - nkv) + lane;
#pragma unroll
              for (int rr = 0; rr < 32; ++rr) {
                const int r = __shfl_sync(0xffffffffu, ridx, rr);
                if (rr < rows_here) kb[static_cast<size_t>(r) * nkv] = __float2bfloat16_rn(stg[rr * 33 + lane]);
              }
            }
          } else {
#pragma unroll
            for (int rr = 0; rr < 32; ++rr) {
              if (rr < rows_here) {
                const float x = stg[rr * 33 + lane];
                if constexpr (EPI == EPI_SWIGLU)
                  epi_elem<EPI>(p, row0 + rr, c, gt[rr], x);
                else
                  epi_elem<EPI>(p, row0 + rr, c, x, 0.f);
              }
            }
          }
        } else {
#pragma unroll
          for (int rr = 0; rr < 32; ++rr) {
            if (rr < rows_here) {
              if constexpr (EPI == EPI_SWIGLU) {
                prow[static_cast<size_t>(rr) * BN + ch * 32 + lane] = gt[rr];
                prow[static_cast<size_t>(rr) * BN + BN / 2 + ch * 32 + lane] = stg[rr * 33 + lane];
              } else {
                prow[static_cast<size_t>(rr) * BN + ch * 32 + lane] = stg[rr * 33 + lane];
              }
            }
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&acce[ab]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if constexpr (CL) {
    if (dsm) {
      cluster_sync_all();  // every split of the cluster is staged
      dsm_reduce<BN, EPI>(p, smem, n, Mt, S);
      cluster_sync_all();  // no CTA leaves while its stage may still be read
    }
  }
}

// Sums the S fp32 partial tiles of a split-K GEMM in split order and runs the
// epilogue.  One thread per (packed row, 8 output columns); all partial loads
// of a thread are issued before the adds.  Returns at once when the GEMM ran
// unsplit (S recomputed from the same n and grid).
// With fold-fill (RESID_SCATTER and p.dep_rng set) the kernel also writes,
// for every folded row r whose source is packed row k, Y[r] = Y[s] +
// (hin[r] - hin[s]) with s = row_idx[k] and Y[s] as stored in bf16; when the
// GEMM ran unsplit it reads Y[s] back and does only the fill.  The folded
// rows of source s are dep_rows[dep_rng[2s] .. dep_rng[2s + 1]).
// Slice j of J of the dependents is filled (the dependents of a source are
// split evenly between J threads when the folded rows far outnumber the
// packed ones, so a few sources with many dependents do not serialise).
// The caller passes the source row s = row_idx[k] and its dependents' range
// rg; the source's input columns go out with the first four folded rows'
// indices, then those rows' inputs (four at a time).
template <int BN, int EPI>
SF_DEV void fill_dependents(const GemmParams& p, int s, int2 rg, int c, const float (&yb)[8], int j = 0, int J = 1) {
  const int len = rg.y - rg.x;
  const int d0 = rg.x + (len * j) / J, d1 = rg.x + (len * (j + 1)) / J;
  if (d1 <= d0) return;
  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(p.Y);
  const uint4 hsv = __ldg(reinterpret_cast<const uint4*>(p.hin + static_cast<size_t>(s) * p.ldy + c));
  for (int j0 = d0; j0 < d1; j0 += 4) {
    uint4 hr[4];
    int rr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) rr[q] = j0 + q < d1 ? p.dep_rows[j0 + q] : -1;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (rr[q] >= 0) hr[q] = __ldg(reinterpret_cast<const uint4*>(p.hin + static_cast<size_t>(rr[q]) * p.ldy + c));
    float hs[8];
    hs[0] = bf16lo(hsv.x); hs[1] = bf16hi(hsv.x); hs[2] = bf16lo(hsv.y); hs[3] = bf16hi(hsv.y);
    hs[4] = bf16lo(hsv.z); hs[5] = bf16hi(hsv.z); hs[6] = bf16lo(hsv.w); hs[7] = bf16hi(hsv.w);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (rr[q] < 0) continue;
      float o[8];
      o[0] = yb[0] + (bf16lo(hr[q].x) - hs[0]); o[1] = yb[1] + (bf16hi(hr[q].x) - hs[1]);
      o[2] = yb[2] + (bf16lo(hr[q].y) - hs[2]); o[3] = yb[3] + (bf16hi(hr[q].y) - hs[3]);
      o[4] = yb[4] + (bf16lo(hr[q].z) - hs[4]); o[5] = yb[5] + (bf16hi(hr[q].z) - hs[5]);
      o[6] = yb[6] + (bf16lo(hr[q].w) - hs[6]); o[7] = yb[7] + (bf16hi(hr[q].w) - hs[7]);
      store_bf16<8>(Y + static_cast<size_t>(rr[q]) * p.ldy + c, o);
    }
  }
}

template <int BN, int EPI>
// (At most 128 registers a thread, so that a block of it fits on an SM beside
// the GEMM CTA it follows and starts early under programmatic launch.)
__global__ void __launch_bounds__(256, 2) splitk_reduce_kernel(const __grid_constant__ GemmParams p, int gemm_grid) {
  const int n_pre = p.n_early && p.n_dev ? __ldcg(p.n_dev) : 0;
  pdl_wait();
  pdl_trigger();
  const int n = p.n_dev ? min(max(p.n_early ? n_pre : p.n_dev[0], 0), p.Mcap) : p.Mcap;
  const Sched sc = get_sched(p.sched, n, p.Nt, p.K / kBK);
  bool fill = false;
  if constexpr (EPI == EPI_RESID_SCATTER) fill = p.dep_rng != nullptr;
  if (sc.S <= 1 && sc.St <= 1 && !fill) return;  // nothing split, nothing to fill
  constexpr int TW = EPI == EPI_SWIGLU ? BN / 2 : BN;   // output columns per tile
  const int groups = (p.Nt * TW) / 8;
  // fold-fill slices: about eight dependents per thread when the folded rows
  // (Mcap - n at most) far outnumber the packed ones
  int J = 1;
  if (fill && n > 0) J = min(16, max(1, (p.Mcap - n + 8 * n - 1) / (8 * n)));
  const long long nk = static_cast<long long>(n) * groups;
  const long long total = nk * J;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int jsl = static_cast<int>(idx / nk);
    const long long kc = idx - static_cast<long long>(jsl) * nk;
    const int k = static_cast<int>(kc / groups);
    const int c = static_cast<int>(kc - static_cast<long long>(k) * groups) * 8;
    const int nt = c / TW, tc = c - nt * TW;
    const int m = k / kBM, row = k - m * kBM;
    int S = 1, slot0 = 0;
    const bool split = tile_split(sc, m, nt, p.Nt, S, slot0);
    // fold-fill: the source row's index first; its dependents' range and the
    // residual go out with the first batch of partials
    int srow = 0;
    int2 rg = make_int2(0, 0);
    uint4 resv = make_uint4(0, 0, 0, 0);
    auto fill_info = [&]() {
      if constexpr (EPI == EPI_RESID_SCATTER) {
        if (fill) {
          rg = reinterpret_cast<const int2*>(p.dep_rng)[srow];
          if (split)
            resv = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.resid) +
                                                        static_cast<size_t>(k) * p.ldr + c));
        }
      }
    };
    if constexpr (EPI == EPI_RESID_SCATTER)
      if (fill) srow = p.row_idx[k];
    if (!split) {
      fill_info();
      if constexpr (EPI == EPI_RESID_SCATTER) {
        // unsplit tile: the GEMM epilogue wrote Y[s]; fill the dependents only
        if (rg.y > rg.x) {
          float yb[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) yb[e] = 0.f;
          add_bf16<8>(static_cast<const __nv_bfloat16*>(p.Y) + static_cast<size_t>(srow) * p.ldy + c, yb);
          fill_dependents<BN, EPI>(p, srow, rg, c, yb, jsl, J);
        }
      }
      continue;
    }
    const float* base = p.partial + static_cast<size_t>(slot0) * kBM * BN + static_cast<size_t>(row) * BN + tc;
    float v[8], u[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = u[e] = 0.f;
#pragma unroll
    for (int s0 = 0; s0 < kMaxSplits; s0 += 8) {
      if (s0 >= S) break;
      float4 a[8][2], b[8][2];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (s0 + q < S) {
          const float4* src = reinterpret_cast<const float4*>(base + static_cast<size_t>(s0 + q) * kBM * BN);
          a[q][0] = __ldcg(src);
          a[q][1] = __ldcg(src + 1);
          if constexpr (EPI == EPI_SWIGLU) {
            b[q][0] = __ldcg(src + BN / 8);
            b[q][1] = __ldcg(src + BN / 8 + 1);
          }
        }
      }
      if (s0 == 0) fill_info();
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (s0 + q < S) {
          v[0] += a[q][0].x; v[1] += a[q][0].y; v[2] += a[q][0].z; v[3] += a[q][0].w;
          v[4] += a[q][1].x; v[5] += a[q][1].y; v[6] += a[q][1].z; v[7] += a[q][1].w;
          if constexpr (EPI == EPI_SWIGLU) {
            u[0] += b[q][0].x; u[1] += b[q][0].y; u[2] += b[q][0].z; u[3] += b[q][0].w;
            u[4] += b[q][1].x; u[5] += b[q][1].y; u[6] += b[q][1].z; u[7] += b[q][1].w;
          }
        }
      }
    }
    // four consecutive threads consumed one 128-byte line of every split
    // (each lane of the quad drops every fourth split's line); not when
    // several fold-fill slices read the same partials
    __syncwarp(__activemask());
    if (J == 1) {
      const float* line = base - (threadIdx.x & 3) * 8;
      for (int s = threadIdx.x & 3; s < S; s += 4) {
        l2_discard_line(line + static_cast<size_t>(s) * kBM * BN);
        if constexpr (EPI == EPI_SWIGLU) l2_discard_line(line + static_cast<size_t>(s) * kBM * BN + BN / 2);
      }
    }
    if constexpr (EPI == EPI_RESID_SCATTER) {
      if (fill) {
        // the residual add and the bf16 rounding of the stored row, then the fill
        v[0] += bf16lo(resv.x); v[1] += bf16hi(resv.x); v[2] += bf16lo(resv.y); v[3] += bf16hi(resv.y);
        v[4] += bf16lo(resv.z); v[5] += bf16hi(resv.z); v[6] += bf16lo(resv.w); v[7] += bf16hi(resv.w);
        if (jsl == 0) store_bf16<8>(static_cast<__nv_bfloat16*>(p.Y) + static_cast<size_t>(srow) * p.ldy + c, v);
        float yb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) yb[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
        fill_dependents<BN, EPI>(p, srow, rg, c, yb, jsl, J);
        continue;
      }
    }
    epi_chunk<EPI, 8>(p, k, nt * TW + tc, v, u);
  }
}

// Down-projection finish with the fold-fill (S9 + S10), in two passes of one
// grid of one CTA per SM (all resident at once).  Pass 1 sums the fp32
// partials of every split tile in split order, adds the residual and writes
// row k to H_out[row_idx[k]] (the GEMM epilogue wrote whole tiles).  After a
// bounded grid barrier, pass 2 gives every folded row r its source's output
// plus its own input difference, H_out[r] = H_out[s] + (H_in[r] - H_in[s])
// with s = src[r], one thread per (row, 8 columns) and four items' loads in
// flight, so a source with many folded rows does not serialise their loads.
// The next kernel may launch only after the barrier (every CTA of this grid
// is resident by then).  With n_early, a thread's first two pass-2 items
// have their sources and input rows read before the wait: src comes from
// the gate/pack kernel and H_in is the layer's input, neither written by the
// GEMM, so after the barrier only the source's output is left to read.
constexpr int kFinThreads = 512;
template <int BN>
__global__ void __launch_bounds__(kFinThreads, 1) down_finish_kernel(const __grid_constant__ GemmParams p) {
  __shared__ volatile int s_flag;
  const int n_pre = p.n_early && p.n_dev ? __ldcg(p.n_dev) : 0;
  const int groups = (p.Nt * BN) / 8;
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long total2 = static_cast<long long>(p.Mcap) * groups;
  constexpr int PRE = 2;
  int pr[PRE], pc[PRE], ps[PRE];
  uint4 phr[PRE], phs[PRE];
  const bool pre = p.n_early != 0;
#pragma unroll
  for (int q = 0; q < PRE; ++q) {
    const long long idx = tid + q * nthr;
    pr[q] = -1;
    ps[q] = -1;
    pc[q] = 0;
    if (pre && idx < total2) {
      pr[q] = static_cast<int>(idx / groups);
      pc[q] = static_cast<int>(idx - static_cast<long long>(pr[q]) * groups) * 8;
      ps[q] = __ldg(p.fill_src + pr[q]);
    }
  }
#pragma unroll
  for (int q = 0; q < PRE; ++q) {
    if (pr[q] >= 0 && ps[q] != pr[q] && ps[q] >= 0 && ps[q] < p.Mcap) {
      phr[q] = __ldg(reinterpret_cast<const uint4*>(p.hin + static_cast<size_t>(pr[q]) * p.ldy + pc[q]));
      phs[q] = __ldg(reinterpret_cast<const uint4*>(p.hin + static_cast<size_t>(ps[q]) * p.ldy + pc[q]));
    }
  }
  pdl_wait();
  const int n = p.n_dev ? min(max(p.n_early ? n_pre : p.n_dev[0], 0), p.Mcap) : p.Mcap;
  const Sched sc = get_sched(p.sched, n, p.Nt, p.K / kBK);
  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(p.Y);
  // ---- pass 1: split tiles
  if (sc.S > 1 || sc.St > 1) {
    const long long total = static_cast<long long>(n) * groups;
    for (long long idx = tid; idx < total; idx += nthr) {
      const int k = static_cast<int>(idx / groups);
      const int c = static_cast<int>(idx - static_cast<long long>(k) * groups) * 8;
      const int nt = c / BN, tc = c - nt * BN;
      const int m = k / kBM, row = k - m * kBM;
      int S = 1, slot0 = 0;
      if (!tile_split(sc, m, nt, p.Nt, S, slot0)) continue;
      const int srow = p.row_idx[k];
      const uint4 resv = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.resid) +
                                                             static_cast<size_t>(k) * p.ldr + c));
      const float* base = p.partial + static_cast<size_t>(slot0) * kBM * BN + static_cast<size_t>(row) * BN + tc;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.f;
      for (int s0 = 0; s0 < S; s0 += 8) {
        float4 a[8][2];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (s0 + q < S) {
            const float4* src = reinterpret_cast<const float4*>(base + static_cast<size_t>(s0 + q) * kBM * BN);
            a[q][0] = __ldcg(src);
            a[q][1] = __ldcg(src + 1);
          }
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (s0 + q < S) {
            v[0] += a[q][0].x; v[1] += a[q][0].y; v[2] += a[q][0].z; v[3] += a[q][0].w;
            v[4] += a[q][1].x; v[5] += a[q][1].y; v[6] += a[q][1].z; v[7] += a[q][1].w;
          }
      }
      // four consecutive threads consumed one 128-byte line of every split
      __syncwarp(__activemask());
      {
        const float* line = base - (threadIdx.x & 3) * 8;
        for (int s = threadIdx.x & 3; s < S; s += 4) l2_discard_line(line + static_cast<size_t>(s) * kBM * BN);
      }
      v[0] += bf16lo(resv.x); v[1] += bf16hi(resv.x); v[2] += bf16lo(resv.y); v[3] += bf16hi(resv.y);
      v[4] += bf16lo(resv.z); v[5] += bf16hi(resv.z); v[6] += bf16lo(resv.w); v[7] += bf16hi(resv.w);
      store_bf16<8>(Y + static_cast<size_t>(srow) * p.ldy + c, v);
    }
  }
  if (!grid_barrier(p.fill_bar, p.status, &s_flag)) return;
  pdl_trigger();
  // ---- pass 2: every folded row from its source's stored output
  for (long long idx0 = tid; idx0 < total2; idx0 += 4 * nthr) {
    const bool first = pre && idx0 == tid;  // items 0 and 1 read before the wait
    int r[4], c[4], s[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const long long idx = idx0 + q * nthr;
      r[q] = -1;
      if (q < PRE && first) {
        r[q] = pr[q];
        c[q] = pc[q];
      } else if (idx < total2) {
        r[q] = static_cast<int>(idx / groups);
        c[q] = static_cast<int>(idx - static_cast<long long>(r[q]) * groups) * 8;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) s[q] = q < PRE && first ? ps[q] : r[q] >= 0 ? __ldg(p.fill_src + r[q]) : -1;
    uint4 ys[4], hr[4], hs[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (r[q] >= 0 && s[q] != r[q] && s[q] >= 0 && s[q] < p.Mcap) {
        ys[q] = __ldcg(reinterpret_cast<const uint4*>(Y + static_cast<size_t>(s[q]) * p.ldy + c[q]));
        if (q < PRE && first) {
          hr[q] = phr[q];
          hs[q] = phs[q];
        } else {
          hr[q] = __ldg(reinterpret_cast<const uint4*>(p.hin + static_cast<size_t>(r[q]) * p.ldy + c[q]));
          hs[q] = __ldg(reinterpret_cast<const uint4*>(p.hin + static_cast<size_t>(s[q]) * p.ldy + c[q]));
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (!(r[q] >= 0 && s[q] != r[q] && s[q] >= 0 && s[q] < p.Mcap)) continue;
      float o[8];
      o[0] = bf16lo(ys[q].x) + (bf16lo(hr[q].x) - bf16lo(hs[q].x));
      o[1] = bf16hi(ys[q].x) + (bf16hi(hr[q].x) - bf16hi(hs[q].x));
      o[2] = bf16lo(ys[q].y) + (bf16lo(hr[q].y) - bf16lo(hs[q].y));
      o[3] = bf16hi(ys[q].y) + (bf16hi(hr[q].y) - bf16hi(hs[q].y));
      o[4] = bf16lo(ys[q].z) + (bf16lo(hr[q].z) - bf16lo(hs[q].z));
      o[5] = bf16hi(ys[q].z) + (bf16hi(hr[q].z) - bf16hi(hs[q].z));
      o[6] = bf16lo(ys[q].w) + (bf16lo(hr[q].w) - bf16lo(hs[q].w));
      o[7] = bf16hi(ys[q].w) + (bf16hi(hr[q].w) - bf16hi(hs[q].w));
      store_bf16<8>(Y + static_cast<size_t>(r[q]) * p.ldy + c[q], o);
    }
  }
}

// Output-projection finish (S6 + S7): one block per packed row k, one thread
// per 8 output columns (GPT groups of 8 when the row is wider than the
// block).  When the GEMM was split, sums the partials in split order, adds the
// residual row H[row_idx[k]] and writes A[k] (bf16); when it was not, A[k] is
// already written by the GEMM epilogue.  Either way the block then
// RMS-normalises the bf16 row: X2[k] = A[k] * g2 / sqrt(mean(A[k]^2) + eps).
// The gains are weights, read before the wait on the GEMM.  With n_early the
// packed-row count and the row index come through L2 before the wait too,
// and so does the residual row (the layer's input, which the GEMM does not
// write); after the wait only the partials' round trip is left.  Without it
// n and the row index come in one round trip after the wait, the residual
// row and the first four splits of every partial in the next.  At most 64
// registers a thread, so that a block fits on an SM beside the GEMM CTA it
// follows and starts early under programmatic launch.
template <int BN, int GPT>
__global__ void __launch_bounds__(512, 2) outproj_finish_kernel(const __grid_constant__ GemmParams p, int gemm_grid,
                                                             const __nv_bfloat16* __restrict__ g2, float eps,
                                                             __nv_bfloat16* __restrict__ X2) {
  __shared__ float s_red[16];
  const int k = blockIdx.x;
  const int groups = p.N / 8;
  const int nthr = static_cast<int>(blockDim.x);
  uint4 gv[GPT];
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    const int gi = threadIdx.x + nthr * j;
    gv[j] = gi < groups ? __ldg(reinterpret_cast<const uint4*>(g2 + gi * 8)) : make_uint4(0, 0, 0, 0);
  }
  // n and this row's index through L2, early, when their producer is known
  // complete (n_early); else after the wait
  const int n_pre = p.n_early && p.n_dev ? __ldcg(p.n_dev) : 0;
  const int r_pre = p.n_early ? __ldcg(p.row_idx + k) : 0;
  // the residual row, early (row_idx[k] is a row of H only for k < n)
  const bool rv_early = p.n_early && k < min(max(n_pre, 0), p.Mcap);
  uint4 rv_pre[GPT];
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    const int gi = threadIdx.x + nthr * j;
    rv_pre[j] = rv_early && gi < groups
                    ? __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.resid) +
                                                           static_cast<size_t>(r_pre) * p.ldr + gi * 8))
                    : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();
  pdl_trigger();
  const int n = p.n_dev ? min(max(p.n_early ? n_pre : p.n_dev[0], 0), p.Mcap) : p.Mcap;
  const int r = p.n_early ? r_pre : p.row_idx[k];  // k < Mcap: in bounds; used only when k < n
  if (k >= n) return;
  const Sched sc = get_sched(p.sched, n, p.Nt, p.K / kBK);
  const int m = k / kBM, row = k - m * kBM;
  __nv_bfloat16* Arow = static_cast<__nv_bfloat16*>(p.Y) + static_cast<size_t>(k) * p.ldy;
  float v[GPT][8];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    const int gi = threadIdx.x + nthr * j;
    if (gi >= groups) break;
    const int c = gi * 8;
    const int nt = c / BN, tc = c - nt * BN;
    int S = 1, slot0 = 0;
    if (tile_split(sc, m, nt, p.Nt, S, slot0)) {
      const uint4 rv = rv_early ? rv_pre[j]
                                : __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.resid) +
                                                                       static_cast<size_t>(r) * p.ldr + c));
      const float* base = p.partial + static_cast<size_t>(slot0) * kBM * BN + static_cast<size_t>(row) * BN + tc;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
      for (int s0 = 0; s0 < S; s0 += 4) {
        float4 a4[4][2];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (s0 + q < S) {
            const float4* src = reinterpret_cast<const float4*>(base + static_cast<size_t>(s0 + q) * kBM * BN);
            a4[q][0] = __ldcg(src);
            a4[q][1] = __ldcg(src + 1);
          }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (s0 + q < S) {
            acc[0] += a4[q][0].x; acc[1] += a4[q][0].y; acc[2] += a4[q][0].z; acc[3] += a4[q][0].w;
            acc[4] += a4[q][1].x; acc[5] += a4[q][1].y; acc[6] += a4[q][1].z; acc[7] += a4[q][1].w;
          }
      }
      acc[0] += bf16lo(rv.x); acc[1] += bf16hi(rv.x); acc[2] += bf16lo(rv.y); acc[3] += bf16hi(rv.y);
      acc[4] += bf16lo(rv.z); acc[5] += bf16hi(rv.z); acc[6] += bf16lo(rv.w); acc[7] += bf16hi(rv.w);
      store_bf16<8>(Arow + c, acc);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[j][e] = __bfloat162float(__float2bfloat16_rn(acc[e]));
    } else {
      const uint4 u = *reinterpret_cast<const uint4*>(Arow + c);
      v[j][0] = bf16lo(u.x); v[j][1] = bf16hi(u.x); v[j][2] = bf16lo(u.y); v[j][3] = bf16hi(u.y);
      v[j][4] = bf16lo(u.z); v[j][5] = bf16hi(u.z); v[j][6] = bf16lo(u.w); v[j][7] = bf16hi(u.w);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(v[j][e], v[j][e], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < nthr / 32; ++w) tot += s_red[w];
  const float inv = rsqrtf(tot / static_cast<float>(p.N) + eps);
#pragma unroll
  for (int j = 0; j < GPT; ++j) {
    const int gi = threadIdx.x + nthr * j;
    if (gi >= groups) break;
    const int c = gi * 8;
    const uint4 gu = gv[j];
    float o[8];
    o[0] = v[j][0] * inv * bf16lo(gu.x); o[1] = v[j][1] * inv * bf16hi(gu.x);
    o[2] = v[j][2] * inv * bf16lo(gu.y); o[3] = v[j][3] * inv * bf16hi(gu.y);
    o[4] = v[j][4] * inv * bf16lo(gu.z); o[5] = v[j][5] * inv * bf16hi(gu.z);
    o[6] = v[j][6] * inv * bf16lo(gu.w); o[7] = v[j][7] * inv * bf16hi(gu.w);
    store_bf16<8>(X2 + static_cast<size_t>(k) * p.N + c, o);
  }
}

// Fills the schedule table of a plain launch on `grid` CTAs (one row per
// m-tile count up to Mcap) and returns whether some n <= Mcap splits a tile,
// i.e. whether the finish kernel has partial tiles to sum.
bool fill_sched(GemmParams& p, int Mcap, int grid) {
  const int KB = p.K / kBK;
  const int mt_max = std::min((Mcap + kBM - 1) / kBM, kSchedRows);
  bool split = false;
  for (int mt = 1; mt <= mt_max; ++mt) {
    const Sched sc = make_sched(mt * kBM, p.Nt, grid, KB);
    p.sched[mt - 1][0] = sc.S;
    p.sched[mt - 1][1] = sc.full;
    p.sched[mt - 1][2] = sc.r;
    p.sched[mt - 1][3] = sc.St;
    p.sched[mt - 1][4] = sc.U;
    split = split || sc.S > 1 || sc.St > 1;
  }
  return split;
}

// Clusters of cs CTAs of the GEMM (one CTA per SM) that can be resident at
// once on the current device, for cs = 2, 4, 8 (queried once per device).
int cluster_capacity(int cs) {
  static int cache[64][kMaxClusterSplit + 1];
  static bool done[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || cs < 2 || cs > kMaxClusterSplit) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    using Cf = Cfg<256>;
    if (cudaFuncSetAttribute(gemm_kernel<256, EPI_STORE, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cf::SMEM_BYTES) == cudaSuccess) {
      for (int c = 2; c <= kMaxClusterSplit; c *= 2)
        cache[dev][c] = max_active_clusters(gemm_kernel<256, EPI_STORE, true>, dim3(kGemmThreads), Cf::SMEM_BYTES, c);
    } else {
      cudaGetLastError();
    }
    done[dev] = true;
  }
  return cache[dev][cs];
}

// SPECFOLD_CLUSTER=0 in the environment turns the clustered split-K off.
bool cluster_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("SPECFOLD_CLUSTER");
    return !(e && e[0] == '0');
  }();
  return on;
}

template <int BN, int EPI>
int run_gemm(const GemmCall& c, cudaStream_t st, const RowNorm* rn, int cs = 0, int cgrid = 0) {
  using Cf = Cfg<BN>;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  int rc = make_map_2d(&p.mapA, c.A, c.Mcap, c.K, c.K, kBM);
  if (rc) return rc;
  int col = 0;
  for (int j = 0; j < c.nb; ++j) {
    rc = make_map_2d(&p.mapB[j], c.b[j], c.b_rows[j], c.K, c.K, BN / 2);
    if (rc) return rc;
    p.col0[j] = col;
    col += c.b_rows[j];
  }
  p.nb = c.nb;
  p.K = c.K;
  p.Mcap = c.Mcap;
  p.N = c.N;
  p.Nt = EPI == EPI_SWIGLU ? c.N / (BN / 2) : c.N / BN;
  p.n_dev = c.n_dev;
  p.Y = c.Y;
  p.ldy = c.ldy;
  p.resid = c.resid;
  p.ldr = c.ldr;
  p.row_idx = c.row_idx;
  p.Yk = c.Yk;
  p.Yv = c.Yv;
  p.n_q = c.n_q;
  p.n_kv = c.n_kv;
  p.hd = c.hd;
  p.g = c.n_kv > 0 ? c.n_q / c.n_kv : 1;
  p.R = c.Mcap;
  if (c.partial_len < gemm_partial_floats()) return SPECFOLD_ECAPACITY;
  p.partial = c.partial;
  p.status = c.status;
  p.n_early = c.n_early ? 1 : 0;
  if constexpr (EPI == EPI_RESID_SCATTER) {
    if (c.dep_rng) {
      if (!c.dep_rows || !c.hin || c.ldy != c.N) return SPECFOLD_EINVAL;
      p.dep_rng = c.dep_rng;
      p.dep_rows = c.dep_rows;
      p.hin = static_cast<const __nv_bfloat16*>(c.hin);
      if (c.fill_src && c.fill_bar) {
        p.fill_src = c.fill_src;
        p.fill_bar = c.fill_bar;
      }
    }
  }

  if (const int rc = smem_limit_once(gemm_kernel<BN, EPI, false>, Cf::SMEM_BYTES)) return rc;
  if (const int rc = smem_limit_once(gemm_kernel<BN, EPI, true>, Cf::SMEM_BYTES)) return rc;
  // schedule table for the plain grid (a clustered launch computes its own
  // split and sums it inside the GEMM)
  const bool any_split = fill_sched(p, c.Mcap, min(num_sms(), kMaxGrid));
  if (cs > 1) {
    // clustered: the splits are summed inside the GEMM
    p.cs = cs;
    launch_kc(gemm_kernel<BN, EPI, true>, dim3(cgrid), dim3(kGemmThreads), Cf::SMEM_BYTES, st, cs, p);
    count_launch();
    if (check_launch()) return SPECFOLD_ECUDA;
    if constexpr (EPI == EPI_RESID_PACKED) {
      if (rn) return launch_rmsnorm_rows(SPECFOLD_BF16, c.Y, nullptr, c.n_dev, c.Mcap, c.N, rn->gain, rn->eps,
                                         rn->out, st);
    }
    return SPECFOLD_OK;
  }
  const int grid = min(num_sms(), kMaxGrid);
  launch_k(gemm_kernel<BN, EPI, false>, dim3(grid), dim3(kGemmThreads), Cf::SMEM_BYTES, st, p);
  count_launch();
  if (check_launch()) return SPECFOLD_ECUDA;
  if constexpr (EPI == EPI_RESID_PACKED) {
    if (rn) {
      const int groups = c.N / 8;
      if (groups > 2 * 512 || c.N % 8) return SPECFOLD_EUNSUPPORTED;
      // one thread per group up to 512 groups, two beyond; with many rows
      // (over four m-tiles) two groups a thread in half as many threads, so
      // more rows' blocks fit on an SM at once (the finish is then bound by
      // its rows in flight, not by one row's latency)
      const int gpt = c.Mcap > 4 * kBM || groups > 512 ? 2 : 1;
      const int threads = std::min(512, ((groups + gpt - 1) / gpt + 31) / 32 * 32);
      const dim3 g(c.Mcap), b(threads);
      const __nv_bfloat16* g2 = static_cast<const __nv_bfloat16*>(rn->gain);
      __nv_bfloat16* x2 = static_cast<__nv_bfloat16*>(rn->out);
      if (gpt == 1)
        launch_k(outproj_finish_kernel<BN, 1>, dim3(g), dim3(b), 0, st, p, grid, g2, rn->eps, x2);
      else
        launch_k(outproj_finish_kernel<BN, 2>, dim3(g), dim3(b), 0, st, p, grid, g2, rn->eps, x2);
      count_launch();
      return check_launch();
    }
  }
  if constexpr (EPI == EPI_RESID_SCATTER) {
    if (p.fill_src) {  // the two-pass finish: split sums, then the fold-fill by folded row
      launch_k(down_finish_kernel<BN>, dim3(grid), dim3(kFinThreads), 0, st, p);
      count_launch();
      return check_launch();
    }
  }
  // the finish kernel sums split tiles; the fold-fill of the down projection
  // runs in it in any case
  if (any_split || p.dep_rng) {
    constexpr int TW = EPI == EPI_SWIGLU ? BN / 2 : BN;
    const long long work = static_cast<long long>(c.Mcap) * (p.Nt * TW / 8);
    const int rgrid = static_cast<int>(std::min<long long>((work + 255) / 256, 8LL * num_sms()));
    launch_k(splitk_reduce_kernel<BN, EPI>, dim3(std::max(rgrid, 1)), dim3(256), 0, st, p, grid);
    count_launch();
    return check_launch();
  }
  return SPECFOLD_OK;
}

struct Plan {
  int BN;
  int cs;     // cluster size, 0 = plain launch
  int grid;   // grid of a clustered launch
};

// Tile width and launch shape.  A clustered split-K launch is planned when
// every n up to Mcap leaves SMs idle (so a split always happens) and its
// clusters cover at least 70 % of the CTAs the plain split would use at one
// m-tile; among those, the plan with most CTAs wins (ties: wider tile).
Plan plan_gemm(int Mcap, int N, int K, bool swiglu, bool ok128, bool ok256) {
  const int grid_nc = min(num_sms(), kMaxGrid);
  Plan plain = {ok256 ? 256 : 128, 0, 0};
  if (!cluster_enabled()) return plain;
  const int Mt_max = (Mcap + kBM - 1) / kBM;
  const int KB = K / kBK;
  const int Nt_plain = swiglu ? N / (plain.BN / 2) : N / plain.BN;
  int S_plain = 1;
  if (Nt_plain < grid_nc) S_plain = std::max(1, std::min({grid_nc / Nt_plain, KB / kMinKbPerSplit, kMaxSplits}));
  const int ctas_plain = Nt_plain * S_plain;
  Plan best = plain;
  int best_ctas = 0;
  for (int BN : {256, 128}) {
    if ((BN == 256 && !ok256) || (BN == 128 && !ok128)) continue;
    const int Nt = swiglu ? N / (BN / 2) : N / BN;
    if (Nt <= 0 || static_cast<long long>(Mt_max) * Nt >= grid_nc) continue;
    for (int cs = kMaxClusterSplit; cs >= 2; cs /= 2) {
      const int G = std::min(cluster_capacity(cs), kMaxGrid / cs) * cs;
      if (G < cs) continue;
      int S = 1;
      for (int d = cs; d > 1; --d)
        if (cs % d == 0 && Nt * d <= G && KB / d >= kMinKbPerSplit) {
          S = d;
          break;
        }
      if (S < 2) continue;
      if (Nt * S > best_ctas) {
        best = {BN, cs, G};
        best_ctas = Nt * S;
      }
    }
  }
  if (best_ctas * 10 < ctas_plain * 7) return plain;
  return best;
}

// Tile width of the residual projections (output and down).  With few
// packed rows the K loop is split to fill the SMs, and every split writes an
// fp32 partial of its whole tile: 128-wide tiles give twice the n-tiles, so
// half the splits and half the partial traffic.  With many rows the GEMM is
// compute-bound and 256-wide tiles read half the shared-memory operand
// bytes per FLOP (a 128-wide tile's MMA runs near the shared-memory read
// rate), so 128 is taken only for at most two m-tiles of rows.
// SPECFOLD_RESID_BN=128 or 256 in the environment fixes the width.
int resid_tile_width(int Mcap, int N) {
  static const int forced = [] {
    const char* e = std::getenv("SPECFOLD_RESID_BN");
    return e ? std::atoi(e) : 0;
  }();
  if (N % 256) return 128;
  if (forced == 128 || forced == 256) return forced;
  return Mcap <= 2 * kBM ? 128 : 256;
}

template <int EPI>
int run_epi(const GemmCall& c, const Plan& pl, cudaStream_t st, const RowNorm* rn = nullptr) {
  return pl.BN == 256 ? run_gemm<256, EPI>(c, st, rn, pl.cs, pl.grid) : run_gemm<128, EPI>(c, st, rn, pl.cs, pl.grid);
}

}  // namespace

// fp32 partial tiles: at most one per persistent CTA (a split happens only
// when tiles * S <= grid).
size_t gemm_partial_floats() { return static_cast<size_t>(kMaxGrid) * kBM * 256; }

int launch_gemm(const GemmCall& c, cudaStream_t st, const RowNorm* rn) {
  if (c.K <= 0 || c.K % kBK || c.Mcap <= 0 || c.N <= 0) return SPECFOLD_EUNSUPPORTED;
  switch (c.epi) {
    case EPI_SWIGLU: {
      if (c.N % 64) return SPECFOLD_EUNSUPPORTED;
      return run_epi<EPI_SWIGLU>(c, plan_gemm(c.Mcap, c.N, c.K, true, true, c.N % 128 == 0), st);
    }
    case EPI_QKV: {
      bool all256 = true;
      for (int j = 0; j < c.nb; ++j) {
        if (c.b_rows[j] % 128) return SPECFOLD_EUNSUPPORTED;
        all256 = all256 && (c.b_rows[j] % 256 == 0);
      }
      if (c.hd % 32) return SPECFOLD_EUNSUPPORTED;
      return run_epi<EPI_QKV>(c, plan_gemm(c.Mcap, c.N, c.K, false, true, all256), st);
    }
    default:
      break;
  }
  if (c.N % 128) return SPECFOLD_EUNSUPPORTED;
  // The residual epilogues keep the plain launch: their split finish is a
  // separate row-parallel kernel that also runs the fused RMSNorm (output
  // projection) or the fold-fill (down projection), and measured faster than
  // the clustered finish, whose whole clusters fit on fewer SMs.
  const Plan plain = {resid_tile_width(c.Mcap, c.N), 0, 0};
  switch (c.epi) {
    case EPI_STORE: return run_epi<EPI_STORE>(c, plan_gemm(c.Mcap, c.N, c.K, false, true, c.N % 256 == 0), st);
    case EPI_RESID_PACKED: return run_epi<EPI_RESID_PACKED>(c, plain, st, rn);
    case EPI_RESID_SCATTER: return run_epi<EPI_RESID_SCATTER>(c, plain, st);
    default: return SPECFOLD_EINVAL;
  }
}

}  // namespace sf

// ===================================================================== //
// specfold_linear_noalloc: the plain GEMM for callers that cannot allocate
// device memory.  Its only scratch, the fp32 split-K partial tiles, lives in
// this file-scope device array, which every GPU that loads the library keeps
// until the process exits.  The persistent grid is capped so that the partial
// tiles of any split fit in it.
// ===================================================================== //
namespace sf {
namespace {

constexpr size_t kNoAllocBytes = static_cast<size_t>(16) << 20;                  // 16 MiB
constexpr int kNoAllocGrid = static_cast<int>(kNoAllocBytes / (kBM * 256 * 4));  // 128 CTAs
constexpr int kNoAllocMaxRows = SPECFOLD_MAX_ROWS;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (in host code the symbol itself is only a host stand-in).
void* noalloc_scratch_ptr() {
  static std::mutex mu;
  static void* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

template <int BN>
int run_linear_noalloc(const void* X, const void* W, int M, int N, int K, void* Y, cudaStream_t st) {
  using Cf = Cfg<BN>;
  const int grid = std::min(num_sms(), kNoAllocGrid);
  // a split writes at most one 128 x BN fp32 tile per CTA of the capped grid
  if (static_cast<size_t>(grid) * kBM * BN * 4 > kNoAllocBytes) return SPECFOLD_ECAPACITY;
  void* scratch = noalloc_scratch_ptr();
  if (!scratch) return SPECFOLD_ECUDA;
  GemmParams p;
  memset(&p, 0, sizeof(p));
  int rc = make_map_2d(&p.mapA, X, M, K, K, kBM);
  if (rc) return rc;
  rc = make_map_2d(&p.mapB[0], W, N, K, K, BN / 2);
  if (rc) return rc;
  p.nb = 1;
  p.K = K;
  p.Mcap = M;
  p.N = N;
  p.Nt = N / BN;
  p.n_dev = nullptr;
  p.Y = Y;
  p.ldy = N;
  p.R = M;
  p.g = 1;
  p.partial = static_cast<float*>(scratch);  // written in full before it is read: nothing to clear
  p.status = nullptr;
  if (const int rc = smem_limit_once(gemm_kernel<BN, EPI_STORE, false>, Cf::SMEM_BYTES)) return rc;
  const bool any_split = fill_sched(p, M, grid);
  launch_k(gemm_kernel<BN, EPI_STORE, false>, dim3(grid), dim3(kGemmThreads), Cf::SMEM_BYTES, st, p);
  count_launch();
  if (check_launch()) return SPECFOLD_ECUDA;
  if (any_split) {
    const long long work = static_cast<long long>(M) * (p.Nt * BN / 8);
    const int rgrid = static_cast<int>(std::min<long long>((work + 255) / 256, 8LL * num_sms()));
    launch_k(splitk_reduce_kernel<BN, EPI_STORE>, dim3(std::max(rgrid, 1)), dim3(256), 0, st, p, grid);
    count_launch();
    return check_launch();
  }
  return SPECFOLD_OK;
}

}  // namespace
}  // namespace sf

extern "C" int specfold_linear_noalloc(int dtype, const void* X, const void* W, int M, int N, int K, void* Y,
                                       void* stream) {
  using namespace sf;
  if (dtype != SPECFOLD_BF16 && dtype != SPECFOLD_F32) return SPECFOLD_EINVAL;
  if (dtype != SPECFOLD_BF16) return SPECFOLD_EUNSUPPORTED;
  if (!X || !W || !Y || M <= 0 || N <= 0 || K <= 0) return SPECFOLD_EINVAL;
  if (M > kNoAllocMaxRows) return SPECFOLD_ECAPACITY;
  if (K % kBK || N % 128) return SPECFOLD_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(Y)) & 15u)
    return SPECFOLD_EALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return N % 256 == 0 ? run_linear_noalloc<256>(X, W, M, N, K, Y, st) : run_linear_noalloc<128>(X, W, M, N, K, Y, st);
}
