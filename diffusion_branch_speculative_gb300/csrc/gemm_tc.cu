// Persistent tcgen05 GEMM for the packed projections of the folded layer
// (QKV, output projection, SwiGLU gate/up, down projection).
//
//   D[k, c] = sum_j A[k, j] * W[c, j]      A: packed rows [Mcap, K] (bf16)
//                                          W: weights [N, K] (bf16, nn.Linear layout)
//
// One CTA per SM loops over work units (m-tile, k-split, n-tile).  The number
// of packed rows n is read on the device, so the decomposition adapts to the
// recompute fraction without a host round trip: when the m x n tiles cannot
// fill the SMs, the K loop is split and the last CTA to finish a tile sums the
// fp32 partials in a fixed order (deterministic) and runs the epilogue.
//
// Roles (192 threads): warp 0 issues TMA loads into a multi-stage ring of
// 128-byte-swizzled tiles; warp 1 allocates TMEM and issues tcgen05.mma
// (M = 128, N = BN, K = 16 per instruction) into one of two TMEM accumulators;
// warps 2-5 read the accumulator back with tcgen05.ld (one row per thread)
// and run the fused epilogue while the next unit accumulates.
#include "sf_device.cuh"
#include "sf_internal.h"

#include <cstring>

namespace sf {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;              // 128 bytes of bf16: one swizzle atom row
constexpr int kGemmThreads = 192;
constexpr int kMaxGrid = 160;        // persistent CTAs (>= SMs of one GB300)
constexpr int kMaxSplits = 16;
constexpr int kMinKbPerSplit = 4;

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
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
  int* counters;
  uint32_t* status;
};

SF_DEV float silu(float x) { return x / (1.f + ex2(-x * 1.4426950408889634f)); }

SF_DEV void store32_bf16(__nv_bfloat16* dst, const float (&v)[32]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    d4[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                       pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}
SF_DEV void add32_bf16(const __nv_bfloat16* src, float (&v)[32]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = __ldg(s4 + q);
    v[8 * q + 0] += bf16lo(u.x); v[8 * q + 1] += bf16hi(u.x);
    v[8 * q + 2] += bf16lo(u.y); v[8 * q + 3] += bf16hi(u.y);
    v[8 * q + 4] += bf16lo(u.z); v[8 * q + 5] += bf16hi(u.z);
    v[8 * q + 6] += bf16lo(u.w); v[8 * q + 7] += bf16hi(u.w);
  }
}

// Epilogue of one 32-column chunk of packed row k.  c = first output column
// (first feature for SWIGLU, where v holds gate and u holds up values).
template <int EPI>
SF_DEV void epi_chunk(const GemmParams& p, int k, int c, float (&v)[32], const float (&u)[32]) {
  __nv_bfloat16* Y = static_cast<__nv_bfloat16*>(p.Y);
  if constexpr (EPI == EPI_STORE) {
    store32_bf16(Y + static_cast<size_t>(k) * p.ldy + c, v);
  } else if constexpr (EPI == EPI_RESID_PACKED) {
    const int r = p.row_idx[k];
    add32_bf16(static_cast<const __nv_bfloat16*>(p.resid) + static_cast<size_t>(r) * p.ldr + c, v);
    store32_bf16(Y + static_cast<size_t>(k) * p.ldy + c, v);
  } else if constexpr (EPI == EPI_RESID_SCATTER) {
    const int r = p.row_idx[k];
    add32_bf16(static_cast<const __nv_bfloat16*>(p.resid) + static_cast<size_t>(k) * p.ldr + c, v);
    store32_bf16(Y + static_cast<size_t>(r) * p.ldy + c, v);
  } else if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = silu(v[e]) * u[e];
    store32_bf16(Y + static_cast<size_t>(k) * p.ldy + c, v);
  } else {  // EPI_QKV
    const int nq = p.n_q * p.hd, nkv = p.n_kv * p.hd;
    if (c < nq) {
      const int head = c / p.hd, j = c - head * p.hd;
      const int hk = head / p.g, hg = head - hk * p.g;
      store32_bf16(Y + ((static_cast<size_t>(hk) * p.R + k) * p.g + hg) * p.hd + j, v);
    } else {
      const int r = p.row_idx[k];
      const bool is_k = c < nq + nkv;
      const int cc = is_k ? c - nq : c - nq - nkv;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(is_k ? p.Yk : p.Yv);
      store32_bf16(dst + static_cast<size_t>(r) * nkv + cc, v);
    }
  }
}

struct Unit {
  int m, s, nt, kb0, kb1, tile;
};

SF_DEV Unit decode(int u, int Mt, int S, int Nt, int KB) {
  Unit w;
  w.m = u % Mt;
  const int rest = u / Mt;
  w.s = rest % S;
  w.nt = rest / S;
  w.kb0 = (w.s * KB) / S;
  w.kb1 = ((w.s + 1) * KB) / S;
  w.tile = w.m * Nt + w.nt;
  return w;
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* accf = bars + 2 * C::STAGES;
  uint64_t* acce = accf + 2;
  uint64_t* drain = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_ok = abort_flag + 1;    // accumulator-ready broadcast
  volatile int* s_last = abort_flag + 2;  // split-K "last CTA of the tile" broadcast

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n_dev ? min(max(p.n_dev[0], 0), p.Mcap) : p.Mcap;
  const int Mt = (n + kBM - 1) / kBM;
  const int tiles = Mt * p.Nt;
  const int KB = p.K / kBK;
  int S = 1;
  if (tiles > 0 && tiles < static_cast<int>(gridDim.x)) {
    S = min(static_cast<int>(gridDim.x) / tiles, KB / kMinKbPerSplit);
    S = max(1, min(S, kMaxSplits));
  }
  const int U = tiles * S;
  if (static_cast<int>(blockIdx.x) >= U) return;

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
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
        const Unit w = decode(u, Mt, S, p.Nt, KB);
        const CUtensorMap* mlo;
        const CUtensorMap* mhi;
        int ylo, yhi;
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
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + st * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          const uint32_t fb = smem_u32(&full[st]);
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
        const Unit w = decode(u, Mt, S, p.Nt, KB);
        const int ab = t & 1;
        if (!mbar_wait(smem_u32(&acce[ab]), ((t >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t dt = tmem_base + ab * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(smem_u32(&full[st]), ph, abort_flag, p.status)) {
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
    const int row = q * 32 + lane;
    uint32_t t = 0;
    for (int u = blockIdx.x; u < U; u += gridDim.x, ++t) {
      const Unit w = decode(u, Mt, S, p.Nt, KB);
      const int ab = t & 1;
      if (et == 0) *s_ok = mbar_wait(smem_u32(&accf[ab]), (t >> 1) & 1, abort_flag, p.status) ? 1 : 0;
      named_bar_sync(1, 128);
      const bool ok = *s_ok != 0;
      named_bar_sync(1, 128);
      if (!ok) break;
      tc_fence_after();
      const int k = w.m * kBM + row;
      const bool valid = k < n;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * BN;
      float* part = p.partial + (static_cast<size_t>(w.tile) * S + w.s) * kBM * BN +
                    static_cast<size_t>(row) * BN;
      if constexpr (EPI == EPI_SWIGLU) {
        for (int ch = 0; ch < BN / 64; ++ch) {
          uint32_t rg[32], ru[32];
          tmem_ld32(tb + ch * 32, rg);
          tmem_ld32(tb + BN / 2 + ch * 32, ru);
          tmem_ld_wait();
          float vg[32], vu[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            vg[e] = __uint_as_float(rg[e]);
            vu[e] = __uint_as_float(ru[e]);
          }
          if (valid) {
            if (S == 1) {
              epi_chunk<EPI>(p, k, w.nt * (BN / 2) + ch * 32, vg, vu);
            } else {
              float4* pg = reinterpret_cast<float4*>(part + ch * 32);
              float4* pu = reinterpret_cast<float4*>(part + BN / 2 + ch * 32);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                pg[e] = make_float4(vg[4 * e], vg[4 * e + 1], vg[4 * e + 2], vg[4 * e + 3]);
                pu[e] = make_float4(vu[4 * e], vu[4 * e + 1], vu[4 * e + 2], vu[4 * e + 3]);
              }
            }
          }
        }
      } else {
        for (int ch = 0; ch < BN / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(tb + ch * 32, r);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
          if (valid) {
            if (S == 1) {
              epi_chunk<EPI>(p, k, w.nt * BN + ch * 32, v, v);
            } else {
              float4* pp = reinterpret_cast<float4*>(part + ch * 32);
#pragma unroll
              for (int e = 0; e < 8; ++e) pp[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&acce[ab]));
      if (S > 1) {
        __threadfence();
        named_bar_sync(1, 128);
        if (et == 0) *s_last = (atomicAdd(&p.counters[w.tile], 1) == S - 1) ? 1 : 0;
        named_bar_sync(1, 128);
        const bool last = *s_last != 0;
        if (last) {
          __threadfence();
          const float* base = p.partial + static_cast<size_t>(w.tile) * S * kBM * BN +
                              static_cast<size_t>(row) * BN;
          if (valid) {
            if constexpr (EPI == EPI_SWIGLU) {
              for (int ch = 0; ch < BN / 64; ++ch) {
                float vg[32], vu[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) vg[e] = vu[e] = 0.f;
                for (int s = 0; s < S; ++s) {
                  const float4* pg = reinterpret_cast<const float4*>(base + static_cast<size_t>(s) * kBM * BN + ch * 32);
                  const float4* pu = reinterpret_cast<const float4*>(base + static_cast<size_t>(s) * kBM * BN + BN / 2 + ch * 32);
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    const float4 a = __ldcg(pg + e), b = __ldcg(pu + e);
                    vg[4 * e] += a.x; vg[4 * e + 1] += a.y; vg[4 * e + 2] += a.z; vg[4 * e + 3] += a.w;
                    vu[4 * e] += b.x; vu[4 * e + 1] += b.y; vu[4 * e + 2] += b.z; vu[4 * e + 3] += b.w;
                  }
                }
                epi_chunk<EPI>(p, k, w.nt * (BN / 2) + ch * 32, vg, vu);
              }
            } else {
              for (int ch = 0; ch < BN / 32; ++ch) {
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0.f;
                for (int s = 0; s < S; ++s) {
                  const float4* pp = reinterpret_cast<const float4*>(base + static_cast<size_t>(s) * kBM * BN + ch * 32);
#pragma unroll
                  for (int e = 0; e < 8; ++e) {
                    const float4 a = __ldcg(pp + e);
                    v[4 * e] += a.x; v[4 * e + 1] += a.y; v[4 * e + 2] += a.z; v[4 * e + 3] += a.w;
                  }
                }
                epi_chunk<EPI>(p, k, w.nt * BN + ch * 32, v, v);
              }
            }
          }
          if (et == 0) p.counters[w.tile] = 0;  // ready for the next call
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN, int EPI>
int run_gemm(const GemmCall& c, cudaStream_t st) {
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
  // the counters must cover every tile this call can have (n = Mcap)
  if (static_cast<long long>((c.Mcap + kBM - 1) / kBM) * p.Nt > c.counters_len) return SPECFOLD_ECAPACITY;
  if (c.partial_len < static_cast<size_t>(kMaxGrid) * kBM * 256) return SPECFOLD_ECAPACITY;
  p.counters = c.counters;
  p.partial = c.partial;
  p.status = c.status;

  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(gemm_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cf::SMEM_BYTES) != cudaSuccess)
      return SPECFOLD_ECUDA;
    attr_done[dev] = 1;
  }
  const int grid = min(num_sms(), kMaxGrid);
  gemm_kernel<BN, EPI><<<grid, kGemmThreads, Cf::SMEM_BYTES, st>>>(p);
  count_launch();
  return check_launch();
}

template <int EPI>
int run_epi(const GemmCall& c, int BN, cudaStream_t st) {
  return BN == 256 ? run_gemm<256, EPI>(c, st) : run_gemm<128, EPI>(c, st);
}

}  // namespace

size_t gemm_partial_floats() { return static_cast<size_t>(kMaxGrid) * kBM * 256; }

int gemm_counters_needed(int Mcap, int N, int epi) {
  const int BN = 128;  // the smaller tile gives the larger count
  const int Nt = epi == EPI_SWIGLU ? N / (BN / 2) : N / BN;
  return ((Mcap + kBM - 1) / kBM) * Nt;
}

int launch_gemm(const GemmCall& c, cudaStream_t st) {
  if (c.K <= 0 || c.K % kBK || c.Mcap <= 0 || c.N <= 0) return SPECFOLD_EUNSUPPORTED;
  int BN = 128;
  switch (c.epi) {
    case EPI_SWIGLU:
      if (c.N % 64) return SPECFOLD_EUNSUPPORTED;
      BN = c.N % 128 == 0 ? 256 : 128;
      return run_epi<EPI_SWIGLU>(c, BN, st);
    case EPI_QKV: {
      bool all256 = true;
      for (int j = 0; j < c.nb; ++j) {
        if (c.b_rows[j] % 128) return SPECFOLD_EUNSUPPORTED;
        all256 = all256 && (c.b_rows[j] % 256 == 0);
      }
      if (c.hd % 32) return SPECFOLD_EUNSUPPORTED;
      return run_epi<EPI_QKV>(c, all256 ? 256 : 128, st);
    }
    default:
      break;
  }
  if (c.N % 128) return SPECFOLD_EUNSUPPORTED;
  BN = c.N % 256 == 0 ? 256 : 128;
  switch (c.epi) {
    case EPI_STORE: return run_epi<EPI_STORE>(c, BN, st);
    case EPI_RESID_PACKED: return run_epi<EPI_RESID_PACKED>(c, BN, st);
    case EPI_RESID_SCATTER: return run_epi<EPI_RESID_SCATTER>(c, BN, st);
    default: return SPECFOLD_EINVAL;
  }
}

}  // namespace sf
