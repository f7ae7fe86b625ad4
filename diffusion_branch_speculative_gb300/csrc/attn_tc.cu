// Folded attention (S5) on the 5th-generation tensor cores.
//
// Work unit = (128 query rows of one KV head, one key range): row m = k*g + j
// of the tile is query head (h*g + j) of packed row k, so a tile mixes the
// GQA group and consecutive packed rows, which may belong to several
// branches.  Keys are streamed in blocks of 128:
//   * the shared prefix (all branches see it) through a 3-D TMA map over the
//     caller's strided view -- never copied per branch;
//   * then the L block keys of every branch present in the tile, gathered
//     through the provenance table (key j of branch b is row src[b*L + j] of
//     the block K/V), with scores of other branches' keys masked.
// A key range is the whole key sequence or, split-KV, one of SP slices whose
// partials a combine kernel merges.  The kernel is persistent: one CTA per SM
// loops over the units of the packed-row count n read on the device, with
// its pipeline running on across units.
// Each key block is worked in two halves of 64 keys, h = 0, 1, that run
// independently within a unit: S_h = Q K_h^T and O_h += P_h V_h run as
// tcgen05.mma into TMEM (two S buffers per half so the next S overlaps the
// softmax, one O accumulator per half), and each half keeps its own running
// max and sum, rescaling O_h in TMEM when its reference max moves.  P_h (bf16)
// goes over the half's own K keys, which S_h has finished with (K is stored
// half by half for that): P is double-buffered with the K/V stages, so the
// softmax of block t never waits for the P V product of block t - 1 except
// to rescale.  At the end of a unit the two halves merge their (O, max, sum)
// the way split-KV partials merge.
//
// Roles (384 threads): warps 0-1 load (TMA for prefix and Q, gathers for
// block keys), warps 2 and 3 issue half 0's and half 1's MMAs (warp 3 also
// owns the TMEM allocation), warps 4-11 softmax: two threads per query row,
// warp w working half (w - 4) / 4 (warp w may only touch TMEM lanes
// 32*(w%4) .. +31), so every SM sub-partition runs one softmax warp of each
// half.  The two threads of a row meet once per unit, to merge.
#include "sf_device.cuh"
#include "sf_internal.h"

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>

namespace sf {
namespace {

constexpr int kAttnThreads = 384;
constexpr int kLoaders = 64;
constexpr int kSmBudget = 160;  // SM count the split sizing plans for (>= one GB300)
constexpr int kAtom = 128 * 128;  // one 128-row x 128-byte swizzle block

struct AttnParams {
  CUtensorMap mapQ;
  CUtensorMap mapK;
  CUtensorMap mapV;
  const __nv_bfloat16* bK;
  const __nv_bfloat16* bV;
  const int32_t* src;
  const int32_t* packed_idx;
  const int32_t* n_dev;
  __nv_bfloat16* O;
  int P, L, R, n_kv, g, n_q;
  float sl2;  // log2(e) / sqrt(hd)
  uint32_t* status;
  // split-KV: SP units share one (query tile, kv head); each writes an
  // unnormalised partial (o, running max m in log2 units, sum l) to slot
  // (h * tiles + x) * SP + z of the live tiles
  int num_sms;
  // paged prefix (table != null): whole 128-key blocks inside one page go
  // through TMA over the pool, the rest through plain gathers
  const int32_t* table;
  int page_size, num_pages, page_tma;
  const __nv_bfloat16* pkp;  // prefix K / V base (pool or contiguous view)
  const __nv_bfloat16* pvp;
  long long k_ts, k_hs, v_ts, v_hs;  // token and head strides, elements
  uint8_t sp_table[1024];            // key-range splits by tile count (see plan_splits)
  float* part_o;    // [slot capacity][128][hd]
  float* part_ml;   // [slot capacity][128][2]
  // CTAs without a unit prefetch into L2 the whole output-projection weight
  // (pf_orb x pf_okb boxes of 128 rows x 64 columns; 0: none), then the
  // first pf_kb k-blocks (64 columns) of every 128-row block of the SwiGLU
  // weights, k-block by k-block (pf_n maps; 0: none)
  CUtensorMap pf_omap;
  int pf_orb, pf_okb;
  CUtensorMap pf_map[2];
  int pf_n, pf_rb, pf_kb;
  int pf_pace_ns;  // pause between one idle CTA's prefetches (queues stay short for the working CTAs' loads)
  int pf_blk_ns;   // expected time of one key block of a working unit (sizes an idle CTA's prefetch budget)
  int pf_delay_ns;  // an idle CTA's pause before its first prefetch
  int n_early;     // n_dev may be read before the programmatic wait (its producer is known complete)
};

// 16-byte asynchronous copy global -> shared that reads `bytes` (16 or 0)
// and zero-fills the rest; completion by cp_async_wait_all in this thread.
SF_DEV void cp_async16_zfill(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
SF_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Number of key-range splits for n packed rows, looked up from a table the
// host fills per launch (sp_table[tiles - 1]; beyond it, no split).  See
// plan_splits for the rule.
constexpr int kSpTable = 1024;
SF_DEV int attn_splits(const AttnParams& p, int rows_total) {
  const int tiles = ((rows_total + 127) / 128) * p.n_kv;
  if (tiles <= 0 || tiles > kSpTable) return 1;
  return p.sp_table[tiles - 1];
}

template <int HD>
struct ACfg {
  static constexpr int NATOM = HD / 64;
  static constexpr int Q_BYTES = kAtom * NATOM;
  static constexpr int KV_BYTES = kAtom * NATOM;  // one K (or V) tile of 128 keys
  // K is stored half by half: keys [64h, 64h + 64) of the block take KH_BYTES
  // at h * KH_BYTES, in NATOM 64-row swizzle atoms of 64 dims each, so half
  // h's product S_h = Q K_h^T reads only its own region
  static constexpr int KH_BYTES = KV_BYTES / 2;
  static constexpr int KH_ATOM = 64 * 128;
  static constexpr int PH_BYTES = kAtom;          // P of one half: 128 rows x 64 keys bf16
  // three K/V stages, so a stage's next keys load while the two before it are
  // still in use (the load of block t must not wait for the P V of block t-1)
  static constexpr int KV_STAGES = 3;
  // P of a half goes over that half's K keys when they have room (hd 128),
  // else into P buffers of their own per stage (hd 64)
  static constexpr bool P_IN_K = PH_BYTES <= KH_BYTES;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = Q_BYTES;  // stage s: K (then P) at +2s*KV, V at +(2s+1)*KV
  static constexpr int OFF_P = OFF_KV + 2 * KV_STAGES * KV_BYTES;
  static constexpr int SMEM_TILES = OFF_P + (P_IN_K ? 0 : KV_STAGES * 2 * PH_BYTES);
  static constexpr int SMEM_BYTES = SMEM_TILES + 1024;  // and the 1024-byte alignment of the base
  static constexpr int p_off(int stage, int h) {
    return P_IN_K ? OFF_KV + 2 * stage * KV_BYTES + h * KH_BYTES : OFF_P + (2 * stage + h) * PH_BYTES;
  }
  // TMEM: S of half h, buffer b at columns (2h + b) * 64; O of half h at
  // COL_O + h * HD
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = 256;
};

// One unit of work (see the file comment) for the live packed-row count.
struct AUnit {
  int x, h, z, m0, b_lo, keys_blk, NB, jb, NT;
  size_t pslot;
};

// The unit's position (tile, head, split): arithmetic only, so the loader can
// start the unit's Q load before the packed-row reads of attn_unit_keys.
SF_DEV AUnit attn_unit_pos(const AttnParams& p, int u, int tiles_x, int SP) {
  AUnit w;
  w.x = u % tiles_x;
  const int rest = u / tiles_x;
  w.h = rest % p.n_kv;
  w.z = rest / p.n_kv;
  w.m0 = w.x * 128;
  w.pslot = (static_cast<size_t>(w.h) * tiles_x + w.x) * SP + w.z;
  return w;
}

// The unit's keys: the branches its rows span and its share of the key blocks.
SF_DEV void attn_unit_keys(const AttnParams& p, AUnit& w, int n, int SP) {
  const int g = p.g, L = p.L, B = p.R / L;
  const int k_lo = w.m0 / g;
  const int k_hi = min(n - 1, (w.m0 + 127) / g);
  w.b_lo = min(max(p.packed_idx[k_lo] / L, 0), B - 1);
  const int b_hi = min(max(p.packed_idx[k_hi] / L, w.b_lo), B - 1);
  w.keys_blk = (b_hi - w.b_lo + 1) * L;
  const int NBP = (p.P + 127) / 128;
  w.NB = NBP + (w.keys_blk + 127) / 128;
  w.jb = (w.z * w.NB) / SP;
  w.NT = ((w.z + 1) * w.NB) / SP - w.jb;
}

SF_DEV AUnit attn_unit(const AttnParams& p, int u, int n, int tiles_x, int SP) {
  AUnit w = attn_unit_pos(p, u, tiles_x, SP);
  attn_unit_keys(p, w, n, SP);
  return w;
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using C = ACfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base; plain pointer arithmetic on the shared array keeps
  // every derived pointer in the shared state space (shared, not generic,
  // loads and stores)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // barriers, flags and the halves' exchange slots in static shared memory
  __shared__ __align__(8) uint64_t bars[25];
  __shared__ uint32_t tmem_slot_s;
  __shared__ volatile int abort_s;
  __shared__ volatile int okflag[C::KV_STAGES];
  // the halves' exchange at the end of a unit, one slot per row (1 KB: the
  // static and dynamic shared memory together sit within a few hundred bytes
  // of the per-block limit at hd 128)
  __shared__ float2 xch[128];
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [KV_STAGES]
  uint64_t* kv_empty = bars + 4;  // [KV_STAGES]: both halves' P V of the block are done
  uint64_t* s_full = bars + 7;    // [half][2]
  uint64_t* s_free = bars + 11;   // [half][2]
  // [half][gi & 1]: two, alternating by block like the S buffers, so that a
  // barrier never runs two phases ahead of the MMA warp that waits on it
  // (the softmax may hand over P of blocks t and t + 1 before that warp, which
  // issued S(t + 1) first, gets to its wait for P(t))
  uint64_t* p_full = bars + 15;
  uint64_t* o_full = bars + 19;   // [half]: one completion per P V product of the half
  uint64_t* q_empty = bars + 21;  // both halves' S products of a unit are done: Q may be replaced
  uint64_t* o_empty = bars + 22;  // the softmax warps have read a unit's outputs
  uint64_t* drain = bars + 23;    // [half]
  uint32_t* tmem_slot = &tmem_slot_s;
  volatile int* abort_flag = &abort_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_pre = p.n_early ? __ldcg(p.n_dev) : 0;
  // Without n_early every thread waits for the previous kernel here.  With
  // it, only the loaders wait, just before the queries and the branch keys,
  // which that kernel (the QKV GEMM) wrote.  Everything else read before
  // that -- n, the packed rows, src -- was written by a kernel that completed
  // before the QKV GEMM's own wait returned, and the prefix is an input of
  // the layer.  (The QKV GEMM and this kernel cannot share an SM, so the
  // TMEM allocation below finds that GEMM's columns already freed.)
  if (!p.n_early) {
    pdl_wait();
    pdl_trigger();
  }
  const int g = p.g, L = p.L;
  const int n = min(max(p.n_early ? n_pre : p.n_dev[0], 0), p.R);
  const int rows_total = n * g;
  const int tiles_x = (rows_total + 127) / 128;
  const int SP = attn_splits(p, rows_total);
  const int U = tiles_x * p.n_kv * SP;
  if (static_cast<int>(blockIdx.x) >= U) {
    if (p.n_early) pdl_trigger();  // it reads nothing the previous kernel wrote
    // no unit for this CTA: its SM would idle through the attention, so it
    // pulls a share of the next GEMMs' weights into L2: the output
    // projection's (needed right after the attention), then the FFN weights'
    // leading k-blocks, in the order the FFN GEMM's CTAs stream them
    if ((p.pf_orb > 0 || p.pf_n > 0) && threadIdx.x == 0) {
      // after the working CTAs' first loads have gone out (a prefetch flood
      // ahead of them delays their first key blocks)
      __nanosleep(p.pf_delay_ns);
      const int idle = static_cast<int>(gridDim.x) - U, me = static_cast<int>(blockIdx.x) - U;
      const int boxes_o = p.pf_orb * p.pf_okb;
      const int boxes = boxes_o + p.pf_n * p.pf_rb * p.pf_kb;
      // Paced only when many idle CTAs share the boxes (a few each): then a
      // burst of prefetches queues ahead of the working CTAs' first loads.
      // With a long share per CTA the pauses would outlast the attention
      // (whose launch ends only when this loop does), so it runs unpaced.
      const int share = (boxes - me + idle - 1) / idle;
      const int pace = share <= 32 ? p.pf_pace_ns : 0;
      // The launch lasts as long as its longest CTA, and one SM issues a
      // box prefetch only every ~0.2 us: a few idle CTAs with the whole
      // share each would outlast the working units.  So each one stops
      // after the boxes that fit in a working unit's expected time (its
      // fixed cost of about four key blocks, then its own key blocks, less
      // the start delay above); together the idle CTAs still cover
      // the leading boxes, in the order the FFN GEMM streams them.
      const int NBu = ((p.P + 127) / 128 + SP) / SP + 1;
      const long long budget_ns = (4LL + NBu) * p.pf_blk_ns - p.pf_delay_ns;
      const int per_box_ns = pace > 0 ? pace + 50 : 250;
      const int cap = budget_ns > 0 ? static_cast<int>(budget_ns / per_box_ns) : 0;
      int issued = 0;
      for (int q = me; q < boxes && issued < cap; q += idle, ++issued) {
        if (pace > 0 && q != me) __nanosleep(pace);
        if (q < boxes_o) {
          const int kb = q / p.pf_orb, rb = q - kb * p.pf_orb;
          tma_prefetch_2d(&p.pf_omap, kb * 64, rb * 128);
          continue;
        }
        const int qf = q - boxes_o;
        const int kb = qf / (p.pf_n * p.pf_rb);
        const int rest = qf - kb * p.pf_n * p.pf_rb;
        const int m = rest / p.pf_rb, rb = rest - m * p.pf_rb;
        tma_prefetch_2d(&p.pf_map[m], kb * 64, rb * 128);
      }
    }
    return;
  }
  const int NBP = (p.P + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int i = 0; i < C::KV_STAGES; ++i) {
      mbar_init(smem_u32(&kv_full[i]), 1);
      mbar_init(smem_u32(&kv_empty[i]), 2);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&s_full[i]), 1);
      mbar_init(smem_u32(&s_free[i]), 128);
    }
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&p_full[i]), 128);
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&o_full[h]), 1);
      mbar_init(smem_u32(&drain[h]), 1);
    }
    mbar_init(smem_u32(q_empty), 2);
    mbar_init(smem_u32(o_empty), 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 3) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint8_t* sQ = smem + C::OFF_Q;

  // Every role walks the same units in the same order; gt counts this CTA's
  // key blocks over all units so far (it sets the ring stage and the phase
  // of every per-block barrier), j its units with keys (Q and O barriers).
  if (warp < 2) {
    // ------------------------------------------------------------ loaders --
    const int lt = threadIdx.x;
    int gt = 0, j = 0;
    int issued_tma = -1, issued_q = -1;
    bool ok = true;
    if (lt == 0) {
      prefetch_tmap(&p.mapQ);
      if (NBP > 0) {
        prefetch_tmap(&p.mapK);
        prefetch_tmap(&p.mapV);
      }
    }
    // the first unit's first prefix block (a fresh stage, no wait for it to
    // empty) goes out before the wait for the previous kernel; its other
    // blocks follow the queries (when that kernel is long done, the queries
    // should not queue behind all three)
    int pre = 0;  // blocks issued before the wait (thread 0 only)
    if (p.n_early && lt == 0 && SP == 1 && NBP > 0 && !p.table) {
      const int h0 = attn_unit_pos(p, blockIdx.x, tiles_x, SP).h;
      uint8_t* sK = smem + C::OFF_KV;  // stage 0, block 0
      uint8_t* sV = sK + C::KV_BYTES;
      const uint32_t fb = smem_u32(&kv_full[0]);
      mbar_arrive_expect_tx(fb, 2 * C::KV_BYTES);
      for (int a = 0; a < C::NATOM; ++a) {
        tma_load_3d(smem_u32(sK + a * C::KH_ATOM), &p.mapK, fb, a * 64, h0, 0);
        tma_load_3d(smem_u32(sK + C::KH_BYTES + a * C::KH_ATOM), &p.mapK, fb, a * 64, h0, 64);
        tma_load_3d(smem_u32(sV + a * kAtom), &p.mapV, fb, a * 64, h0, 0);
      }
      issued_tma = 0;
      pre = 1;
    }
    if (p.n_early) {
      pdl_wait();
      pdl_trigger();  // (as every thread does at the top without n_early)
    }
    for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
      AUnit w = attn_unit_pos(p, u, tiles_x, SP);
      const int h = w.h;
      // a unit without keys (more splits than key blocks) loads nothing; NT
      // is 0 only when SP > NB, and NB >= NBP + 1 always
      const bool may_be_empty = SP > NBP + 1;
      if (lt == 0 && !may_be_empty) {
        // the previous unit's S products must be done with the Q buffer
        if (j == 0 || mbar_wait(smem_u32(q_empty), (j - 1) & 1, abort_flag, p.status, kWaitLimitNs, kSiteAttnQEmpty)) {
          mbar_arrive_expect_tx(smem_u32(q_full), C::Q_BYTES);
          for (int a = 0; a < C::NATOM; ++a)
            tma_load_2d(smem_u32(sQ + a * kAtom), &p.mapQ, smem_u32(q_full), a * 64, h * p.R * g + w.m0);
          issued_q = j;
        }
      }
      // An unsplit unit starts with the whole prefix, so its first block goes
      // out before the packed-row reads that size its block keys (their
      // round trip then overlaps that block's load)
      bool keys_known = SP > 1 || NBP == 0;
      if (keys_known) {
        attn_unit_keys(p, w, n, SP);
      } else {
        w.jb = 0;
        w.NT = NBP + 1;  // a lower bound: at least one block of branch keys follows
      }
      if (w.NT == 0) continue;
      if (lt == 0 && may_be_empty) {
        if (j == 0 || mbar_wait(smem_u32(q_empty), (j - 1) & 1, abort_flag, p.status, kWaitLimitNs, kSiteAttnQEmpty)) {
          mbar_arrive_expect_tx(smem_u32(q_full), C::Q_BYTES);
          for (int a = 0; a < C::NATOM; ++a)
            tma_load_2d(smem_u32(sQ + a * kAtom), &p.mapQ, smem_u32(q_full), a * 64, h * p.R * g + w.m0);
          issued_q = j;
        }
      }
      for (int t = 0; t < w.NT; ++t, ++gt) {
        if (!keys_known && t == 1) {
          attn_unit_keys(p, w, n, SP);  // the same NT every other role computed
          keys_known = true;
        }
        const int jblk = w.jb + t;
        const int st = gt % C::KV_STAGES;
        const bool early_blk = gt < pre;  // issued before the wait (thread 0 only)
        if (lt == 0)
          okflag[st] = early_blk || mbar_wait(smem_u32(&kv_empty[st]), ((gt / C::KV_STAGES) & 1) ^ 1, abort_flag, p.status,
                                              kWaitLimitNs, kSiteAttnKvEmpty) ? 1 : 0;
        named_bar_sync(1, kLoaders);
        if (!okflag[st]) {
          ok = false;
          break;
        }
        uint8_t* sK = smem + C::OFF_KV + (2 * st) * C::KV_BYTES;
        uint8_t* sV = sK + C::KV_BYTES;
        // prefix blocks go through TMA unless paged with the block not inside
        // one page or not whole (pool tokens past P may hold anything)
        const bool use_tma = jblk < NBP && (!p.table || (p.page_tma && (jblk + 1) * 128 <= p.P));
        if (use_tma) {
          if (lt == 0 && !early_blk) {
            int z = jblk * 128;
            if (p.table) {
              const int page = p.table[(jblk * 128) / p.page_size];
              if (page >= 0 && page < p.num_pages) {
                z = page * p.page_size + (jblk * 128) % p.page_size;
              } else {
                z = p.num_pages * p.page_size;  // wholly past the pool: the box reads zeros
                atomicOr(p.status, SPECFOLD_DEV_BAD_PAGE);
              }
            }
            const uint32_t fb = smem_u32(&kv_full[st]);
            mbar_arrive_expect_tx(fb, 2 * C::KV_BYTES);
            for (int a = 0; a < C::NATOM; ++a) {
              // K half by half (64-token boxes), V whole (128-token boxes)
              tma_load_3d(smem_u32(sK + a * C::KH_ATOM), &p.mapK, fb, a * 64, h, z);
              tma_load_3d(smem_u32(sK + C::KH_BYTES + a * C::KH_ATOM), &p.mapK, fb, a * 64, h, z + 64);
              tma_load_3d(smem_u32(sV + a * kAtom), &p.mapV, fb, a * 64, h, z);
            }
            issued_tma = gt;
          }
        } else {
          // Gathered rows: first every row's source (the page table or src
          // read, one round trip for all of this thread's rows), then each
          // 16-byte chunk copied asynchronously straight to its swizzled
          // place, zero-filled for a missing row, all in flight at once.
          constexpr int RPT = 128 / kLoaders;  // rows per thread
          const __nv_bfloat16* krow[RPT];
          const __nv_bfloat16* vrow[RPT];
#pragma unroll
          for (int q = 0; q < RPT; ++q) {
            const int kr = lt + q * kLoaders;
            krow[q] = vrow[q] = nullptr;
            if (jblk < NBP) {  // paged prefix token
              const int tk = jblk * 128 + kr;
              if (tk < p.P) {
                const int page = p.table[tk / p.page_size];
                if (page >= 0 && page < p.num_pages) {
                  const size_t tok = static_cast<size_t>(page) * p.page_size + tk % p.page_size;
                  krow[q] = p.pkp + tok * p.k_ts + static_cast<size_t>(h) * p.k_hs;
                  vrow[q] = p.pvp + tok * p.v_ts + static_cast<size_t>(h) * p.v_hs;
                } else {
                  atomicOr(p.status, SPECFOLD_DEV_BAD_PAGE);
                }
              }
            } else {
              const int e = (jblk - NBP) * 128 + kr;
              if (e < w.keys_blk) {
                const int b = w.b_lo + e / L;
                const int s = p.src[b * L + (e - (e / L) * L)];
                if (s >= 0 && s < p.R) {  // an invalid source reads as a zero key and value
                  const size_t off = (static_cast<size_t>(s) * p.n_kv + h) * HD;
                  krow[q] = p.bK + off;
                  vrow[q] = p.bV + off;
                }
              }
            }
          }
#pragma unroll
          for (int q = 0; q < RPT; ++q) {
            const int kr = lt + q * kLoaders;
            const int kh = kr >> 6, kq = kr & 63;  // half of the block and row within it
            const uint32_t nk = krow[q] ? 16u : 0u, nv = vrow[q] ? 16u : 0u;
            const __nv_bfloat16* ks = krow[q] ? krow[q] : p.bK;  // any valid address when nothing is read
            const __nv_bfloat16* vs = vrow[q] ? vrow[q] : p.bV;
#pragma unroll
            for (int c16 = 0; c16 < HD / 8; ++c16) {
              const int sw = ((c16 & 7) ^ (kr & 7)) << 4;
              cp_async16_zfill(smem_u32(sK + kh * C::KH_BYTES + (c16 >> 3) * C::KH_ATOM + kq * 128 + sw), ks + c16 * 8, nk);
              cp_async16_zfill(smem_u32(sV + (c16 >> 3) * kAtom + kr * 128 + sw), vs + c16 * 8, nv);
            }
          }
          cp_async_wait_all();
          fence_proxy_async_smem();
          named_bar_sync(1, kLoaders);
          if (lt == 0) mbar_arrive(smem_u32(&kv_full[st]));
        }
      }
      ++j;
    }
    if (lt == 0 && *abort_flag) {
      // let the copies already issued land before the CTA exits
      int never = 0;
      if (issued_tma >= 0)
        mbar_wait(smem_u32(&kv_full[issued_tma % C::KV_STAGES]), (issued_tma / C::KV_STAGES) & 1, &never, nullptr,
                  10000000ull);
      if (issued_q >= 0) mbar_wait(smem_u32(q_full), issued_q & 1, &never, nullptr, 10000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax --
    // Two threads per query row: half hf of the row owns keys [64 hf, 64 hf +
    // 64) of every block, with its own S products, its own output
    // accumulator O_hf in TMEM (P_hf V_hf with accumulate), its own reference
    // max m and sum l: within a unit the halves never wait for each other.
    // A half raises m -- and rescales its O in place -- only when its max
    // grows by more than 2^8, so its probabilities stay below 2^8.  At the end
    // of the unit the halves meet once and merge: with M = max(m_0, m_1) and
    // w_h = 2^(m_h - M), the row's output is (w_0 O_0 + w_1 O_1) / (w_0 l_0 +
    // w_1 l_1), half hf writing output columns [hf HD/2, (hf + 1) HD/2).
    const int qw = warp & 3;
    const int hf = (warp - 4) >> 2;
    const int row = qw * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    constexpr int OH = HD / 2;  // output columns a thread writes
    const uint32_t to_own = tmem + lane_off + C::COL_O + hf * HD;
    const int pair_bar = 2 + qw;  // named barrier of the two warps sharing these rows
    int gt = 0, j = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
      const AUnit w = attn_unit(p, u, n, tiles_x, SP);
      if (w.NT == 0) {  // empty key range: a neutral partial
        float* po = p.part_o + (w.pslot * 128 + row) * HD + hf * OH;
        for (int c = 0; c < OH; c += 4) *reinterpret_cast<float4*>(po + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (hf == 0) {
          p.part_ml[(w.pslot * 128 + row) * 2] = -INFINITY;
          p.part_ml[(w.pslot * 128 + row) * 2 + 1] = 0.f;
        }
        continue;
      }
      const int h = w.h;
      const int m = w.m0 + row;
      const bool valid = m < rows_total;
      const int k = valid ? m / g : 0;
      const int hg = m - (m / g) * g;
      const int my_b = valid ? p.packed_idx[k] / L : -2;
      float m_ref = -INFINITY, l = 0.f;
      for (int t = 0; t < w.NT; ++t) {
        const int gi = gt + t;
        const int jblk = w.jb + t;
        const int sb = gi & 1;
        const bool prefix = jblk < NBP;
        // every wait's outcome is made warp-uniform: a lane whose wait ran out
        // takes its whole warp along
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[2 * hf + sb]), (gi >> 1) & 1, abort_flag, p.status, kWaitLimitNs,
                                                         kSiteAttnSFull))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int key0 = jblk * 128 + hf * 64;  // first key of this half
        const uint32_t ts = tmem + lane_off + (2 * hf + sb) * 64;
        uint32_t sv[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_ld32(ts + c * 32, sv[c]);
        // visibility of the 64 keys as two 32-bit masks (bit e of km[c]: key
        // 32c + e of the half): prefix keys below P; block keys of this row's
        // own branch, one run of L keys
        uint32_t km[2];
        {
          int lo, hi;  // visible keys [lo, hi) relative to this half's first key
          if (prefix) {
            lo = 0;
            hi = p.P - key0;
          } else {
            lo = (my_b - w.b_lo) * L - ((jblk - NBP) * 128 + hf * 64);
            hi = lo + L;
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int a0 = max(lo - c * 32, 0), a1 = min(hi - c * 32, 32);
            km[c] = a1 > a0 ? ((a1 >= 32 ? 0xffffffffu : ((1u << a1) - 1u)) & ~((1u << a0) - 1u)) : 0u;
          }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_ld_wait(sv[c]);
        tc_fence_before();
        mbar_arrive(smem_u32(&s_free[2 * hf + sb]));   // the S buffer may be refilled now
        // a whole prefix half-block needs no mask; eight independent max chains
        const bool allv = prefix && p.P - key0 >= 64;
        float mx8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx8[q] = -INFINITY;
        if (allv) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], __uint_as_float(sv[c][e]));
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              mx8[e & 7] = fmaxf(mx8[e & 7], ((km[c] >> e) & 1u) ? __uint_as_float(sv[c][e]) : -INFINITY);
        }
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_new = fmaxf(m_ref, mx * p.sl2);
        float alpha = 1.f;
        bool rescale = false;
        if (m_ref == -INFINITY) {
          m_ref = m_new;               // nothing accumulated yet (every earlier p was 0)
        } else if (m_new > m_ref + 8.f) {
          alpha = ex2(m_ref - m_new);
          m_ref = m_new;
          rescale = true;
        }
        l *= alpha;
        // O_hf may only be rescaled once it holds the previous block's P V
        bool rescale_waited = false;
        if (t >= 1 && __any_sync(0xffffffffu, rescale)) {
          rescale_waited = true;
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&o_full[hf]), (gi - 1) & 1, abort_flag, p.status, kWaitLimitNs, kSiteAttnRescale))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(to_own + c * 32, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(to_own + c * 32, r);
          }
          tmem_st_wait();
        }
        // probabilities -> bf16 P_hf tile (128 rows x 64 keys, K-major,
        // 128-byte swizzle); the sum in four independent partial sums
        uint8_t* sP = smem + C::p_off(gi % C::KV_STAGES, hf);
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
          if (allv) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float x0 = ex2(fmaf(__uint_as_float(sv[c][e]), p.sl2, -m_ref));
              const float x1 = ex2(fmaf(__uint_as_float(sv[c][e + 1]), p.sl2, -m_ref));
              ls[(e >> 1) & 3] += x0 + x1;
              pk[e / 2] = pack_bf16x2(x0, x1);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float pv[2];
#pragma unroll
              for (int uu = 0; uu < 2; ++uu) {
                const float x = ex2(fmaf(__uint_as_float(sv[c][e + uu]), p.sl2, -m_ref));
                pv[uu] = ((km[c] >> (e + uu)) & 1u) ? x : 0.f;
              }
              ls[(e >> 1) & 3] += pv[0] + pv[1];
              pk[e / 2] = pack_bf16x2(pv[0], pv[1]);
            }
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int kc = c * 4 + q4;  // 8-key chunk of the half, 0..7
            const int off = row * 128 + ((kc ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(sP + off) = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
          }
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // A parity wait is exact only while its barrier cannot run two phases
        // ahead.  o_full completes once per P V; P V of block gi - 2 is done
        // once S(gi) is (the MMA warp issues S(gi) after it), and P V of block
        // gi cannot start before this thread's p_full below.  So the wait for
        // P V of block gi - 1 is exact here, and the unit's last block takes
        // it before handing over its P: afterwards only the last P V is out,
        // and the wait for it after the loop is exact too.
        if (t == w.NT - 1 && t >= 1 && !rescale_waited) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&o_full[hf]), (gi - 1) & 1, abort_flag, p.status, kWaitLimitNs, kSiteAttnLastP))) {
            ok = false;
            break;
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&p_full[2 * hf + sb]));
      }
      // the half's last P V product (the one before it is done, see above)
      const int glast = gt + w.NT - 1;
      const bool oku = ok && mbar_wait(smem_u32(&o_full[hf]), glast & 1, abort_flag, p.status, kWaitLimitNs, kSiteAttnEnd);
      // the halves' meeting at the end of the unit: both leave together or
      // neither (a wait that ran out must not strand the other half at a
      // barrier).  Half 1 hands its (m, l) to half 0, which computes the merge
      // weights w_h = 2^(m_h - M) (divided by the row's sum when the output is
      // final) and hands half 1 its pair back.  The first barrier also orders
      // half 0's reads of the previous unit's hand-back before this write.
      if (hf == 1) xch[row] = make_float2(m_ref, l);
      tc_fence_before();
      __syncwarp();
      if (!named_bar_and(pair_bar, 64, oku)) { ok = false; break; }
      tc_fence_after();
      float a0 = 0.f, a1 = 0.f, M = 0.f, lrow = 0.f;
      if (hf == 0) {
        const float2 o1 = xch[row];
        M = fmaxf(m_ref, o1.x);
        const float w0 = m_ref == -INFINITY ? 0.f : ex2(m_ref - M);
        const float w1 = o1.x == -INFINITY ? 0.f : ex2(o1.x - M);
        lrow = w0 * l + w1 * o1.y;
        const float sc = SP > 1 ? 1.f : 1.f / lrow;  // split: the partial stays unnormalised
        a0 = w0 * sc;
        a1 = w1 * sc;
        xch[row] = make_float2(a0, a1);
      }
      named_bar_sync(pair_bar, 64);
      if (hf == 1) {
        const float2 f = xch[row];
        a0 = f.x;
        a1 = f.y;
      }
      const uint32_t t0 = tmem + lane_off + C::COL_O + hf * OH;  // columns [hf OH, (hf + 1) OH) of O_0
      const uint32_t t1 = t0 + HD;                                // ... and of O_1
      if (SP > 1) {
        float* po = p.part_o + (w.pslot * 128 + row) * HD + hf * OH;
#pragma unroll
        for (int c = 0; c < OH / 32; ++c) {
          uint32_t r0[32], r1[32];
          tmem_ld32(t0 + c * 32, r0);
          tmem_ld32(t1 + c * 32, r1);
          tmem_ld_wait(r0);
          tmem_ld_wait(r1);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              o[e] = a0 * __uint_as_float(r0[4 * q4 + e]) + a1 * __uint_as_float(r1[4 * q4 + e]);
            reinterpret_cast<float4*>(po + c * 32)[q4] = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
        if (hf == 0) {
          p.part_ml[(w.pslot * 128 + row) * 2] = M;
          p.part_ml[(w.pslot * 128 + row) * 2 + 1] = lrow;
        }
      } else {
        uint4* dst = reinterpret_cast<uint4*>(p.O + static_cast<size_t>(k) * (p.n_q * HD) +
                                              static_cast<size_t>(h * g + hg) * HD + hf * OH);
#pragma unroll
        for (int c = 0; c < OH / 32; ++c) {
          uint32_t r0[32], r1[32];
          tmem_ld32(t0 + c * 32, r0);
          tmem_ld32(t1 + c * 32, r1);
          tmem_ld_wait(r0);
          tmem_ld_wait(r1);
          if (valid) {
            auto ov = [&](int e) { return a0 * __uint_as_float(r0[e]) + a1 * __uint_as_float(r1[e]); };
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8)
              dst[c * 4 + q8] = make_uint4(pack_bf16x2(ov(8 * q8), ov(8 * q8 + 1)), pack_bf16x2(ov(8 * q8 + 2), ov(8 * q8 + 3)),
                                           pack_bf16x2(ov(8 * q8 + 4), ov(8 * q8 + 5)),
                                           pack_bf16x2(ov(8 * q8 + 6), ov(8 * q8 + 7)));
          }
        }
      }
      // the accumulators are free for the next unit's first P V products
      tc_fence_before();
      mbar_arrive(smem_u32(o_empty));
      gt += w.NT;
      ++j;
    }
  } else {
    // ---------------------------------------------------------------- MMA --
    // warp 2 issues half 0's products, warp 3 half 1's: S_h = Q K_h^T
    // (N = 64) into S buffer (h, gi & 1) and O_h += P_h V_h (K = 64 keys)
    const int hm = warp - 2;
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 64, false);
      constexpr uint32_t idPV = idesc_bf16_f32(128, HD, true);
      const uint32_t aQ = smem_u32(sQ);
      const uint32_t tO = tmem + C::COL_O + hm * HD;
      int gt = 0, j = 0;
      bool ok = true;
      // P_h V_h of key block gi (first: the unit's first block, which
      // overwrites O_h: the softmax warps have read the previous unit's
      // outputs by then, see the o_empty wait below)
      auto issue_pv = [&](int gi, bool first) -> bool {
        if (!mbar_wait(smem_u32(&p_full[2 * hm + (gi & 1)]), (gi >> 1) & 1, abort_flag, p.status, kWaitLimitNs,
                       kSiteAttnPFull))
          return false;
        tc_fence_after();
        const int kst = gi % C::KV_STAGES;
        const uint32_t aP = smem_u32(smem + C::p_off(kst, hm));
        const uint32_t aV = smem_u32(smem + C::OFF_KV + (2 * kst + 1) * C::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc_mma_f16(tO, sdesc_sw128(aP + kk * 32, 16, 1024), sdesc_sw128(aV + (4 * hm + kk) * 2048, kAtom, 1024),
                     idPV, (!first || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&o_full[hm]));
        tc_commit(smem_u32(&kv_empty[kst]));
        return true;
      };
      for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
        const AUnit w = attn_unit(p, u, n, tiles_x, SP);
        if (w.NT == 0) continue;
        if (!mbar_wait(smem_u32(q_full), j & 1, abort_flag, p.status, kWaitLimitNs, kSiteAttnQFull)) break;
        for (int t = 0; t < w.NT && ok; ++t) {
          const int gi = gt + t;
          const int sb = gi & 1;              // S buffer
          const int kst = gi % C::KV_STAGES;  // K/V stage
          if (!mbar_wait(smem_u32(&kv_full[kst]), (gi / C::KV_STAGES) & 1, abort_flag, p.status, kWaitLimitNs,
                         kSiteAttnKvFull)) { ok = false; break; }
          if (!mbar_wait(smem_u32(&s_free[2 * hm + sb]), ((gi >> 1) & 1) ^ 1, abort_flag, p.status, kWaitLimitNs,
                         kSiteAttnSFree)) { ok = false; break; }
          // Before the unit's second S (or its only P V): both halves have
          // read the previous unit's outputs.  Waiting here, and not just
          // before the first P V, keeps p_full exact: with S(1) not yet
          // issued, the softmax can hand over at most block 0's P before the
          // p_full wait below.
          if (t == 1 && j >= 1 && !mbar_wait(smem_u32(o_empty), (j - 1) & 1, abort_flag, p.status, kWaitLimitNs, kSiteAttnOEmpty)) { ok = false; break; }
          tc_fence_after();
          const uint32_t aK = smem_u32(smem + C::OFF_KV + (2 * kst) * C::KV_BYTES + hm * C::KH_BYTES);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            tc_mma_f16(tmem + (2 * hm + sb) * 64,
                       sdesc_sw128(aQ + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024),
                       sdesc_sw128(aK + (kk >> 2) * C::KH_ATOM + (kk & 3) * 32, 16, 1024), idS, kk > 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&s_full[2 * hm + sb]));
          if (t == w.NT - 1) tc_commit(smem_u32(q_empty));  // Q is read by no later product of this unit
          if (t >= 1 && !issue_pv(gi - 1, t == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (w.NT == 1 && j >= 1 && !mbar_wait(smem_u32(o_empty), (j - 1) & 1, abort_flag, p.status, kWaitLimitNs, kSiteAttnOEmpty)) break;
        if (!issue_pv(gt + w.NT - 1, w.NT == 1)) break;
        gt += w.NT;
        ++j;
      }
      tc_commit(smem_u32(&drain[hm]));
      int never = 0;
      mbar_wait(smem_u32(&drain[hm]), 0, &never, nullptr, 10000000ull);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Merges the split-KV partials: for each (query row, kv head, 8 dims),
// O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s with M = max_s m_s.
template <int HD>
__global__ void __launch_bounds__(256) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  pdl_wait();
  pdl_trigger();
  const int n = min(max(p.n_dev[0], 0), p.R);
  const int rows_total = n * p.g;
  const int SP = attn_splits(p, rows_total);
  if (SP <= 1) return;
  const int tiles_x = (rows_total + 127) / 128;
  constexpr int DG = HD / 8;
  const long long total = static_cast<long long>(rows_total) * p.n_kv * DG;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int dg = static_cast<int>(idx % DG);
    const long long rest = idx / DG;
    const int m = static_cast<int>(rest % rows_total);
    const int h = static_cast<int>(rest / rows_total);
    const int row = m & 127;
    const size_t pb = (static_cast<size_t>(h) * tiles_x + (m >> 7)) * SP;
    // every load of the row is issued before any arithmetic
    float mz[16], lz[16];
    float4 oa[16], ob[16];
#pragma unroll
    for (int z = 0; z < 16; ++z) {
      if (z < SP) {
        const float* ml = p.part_ml + ((pb + z) * 128 + row) * 2;
        mz[z] = __ldcg(ml);
        lz[z] = __ldcg(ml + 1);
        const float4* src = reinterpret_cast<const float4*>(p.part_o + ((pb + z) * 128 + row) * HD + dg * 8);
        oa[z] = __ldcg(src);
        ob[z] = __ldcg(src + 1);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int z = 0; z < 16; ++z)
      if (z < SP) M = fmaxf(M, mz[z]);
    float l = 0.f, acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
    for (int z = 0; z < 16; ++z) {
      if (z < SP && mz[z] != -INFINITY) {
        const float wz = ex2(mz[z] - M);
        l = fmaf(lz[z], wz, l);
        acc[0] = fmaf(oa[z].x, wz, acc[0]); acc[1] = fmaf(oa[z].y, wz, acc[1]);
        acc[2] = fmaf(oa[z].z, wz, acc[2]); acc[3] = fmaf(oa[z].w, wz, acc[3]);
        acc[4] = fmaf(ob[z].x, wz, acc[4]); acc[5] = fmaf(ob[z].y, wz, acc[5]);
        acc[6] = fmaf(ob[z].z, wz, acc[6]); acc[7] = fmaf(ob[z].w, wz, acc[7]);
      }
    }
    // four consecutive threads consumed one 128-byte line of every split's o
    __syncwarp(__activemask());
    for (int z = dg & 3; z < SP; z += 4) l2_discard_line(p.part_o + ((pb + z) * 128 + row) * HD + (dg & ~3) * 8);
    const float inv = 1.f / l;
    const int k = m / p.g, hg = m - k * p.g;
    uint4* dst = reinterpret_cast<uint4*>(p.O + static_cast<size_t>(k) * (p.n_q * HD) +
                                          static_cast<size_t>(h * p.g + hg) * HD + dg * 8);
    *dst = make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                      pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
  }
}

// Split count for `tiles` (query tile, KV head) pairs: with one CTA per SM,
// S splits cost about ceil(tiles * S / SMs) waves, each unit paying a fixed
// cost (first loads, the write-out of its output or partial, which the
// softmax warps do in series with their next unit: about four key blocks)
// plus its share
// nb / S of the key blocks, and a split adds the combine launch (about
// `combine` key blocks); the S with the least cost (the smallest on a near
// tie), at most one more than the key blocks (the block keys may span two)
// and at most sp_lim.
int plan_splits(int tiles, int sp_lim, int num_sms, int P, float combine) {
  const float nb = static_cast<float>((P + 127) / 128 + 1);
  int best = 1;
  constexpr float kUnit = 4.f;
  float best_t = static_cast<float>((tiles + num_sms - 1) / num_sms) * (kUnit + nb);
  for (int sp = 2; sp <= sp_lim && sp <= nb + 1; ++sp) {
    const float t = static_cast<float>((tiles * sp + num_sms - 1) / num_sms) * (kUnit + nb / sp) + combine;
    if (t < best_t * 0.97f) {
      best = sp;
      best_t = t;
    }
  }
  return best;
}

// SPECFOLD_FFN_PREFETCH=0 in the environment turns the weight prefetch of the
// attention's idle CTAs off; SPECFOLD_FFN_PREFETCH_MB sets its FFN share
// (default 40 MB); SPECFOLD_PREFETCH_WO=1 adds the output projection's weight
// ahead of it (off by default: at the 7B layer it slowed the attention by
// more than it saved in the projection); SPECFOLD_PREFETCH_PACE_NS sets the
// pause between one idle CTA's prefetches (default 400 ns), and
// SPECFOLD_PREFETCH_BLOCK_NS the expected time of one key block of a working
// unit (default 1500 ns), which bounds how long an idle CTA keeps
// prefetching; SPECFOLD_PREFETCH_DELAY_NS the pause before an idle CTA's
// first prefetch (default 3000 ns).
static int env_int(const char* name, int dflt) {
  const char* e = std::getenv(name);
  return e ? std::atoi(e) : dflt;
}
bool ffn_prefetch_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("SPECFOLD_FFN_PREFETCH");
    return !(e && e[0] == '0');
  }();
  return on;
}

// Cost of the combine launch in key blocks: writing and reading back the
// fp32 partials plus a launch (SPECFOLD_ATTN_COMBINE_COST overrides it;
// SPECFOLD_ATTN_SPLITS=k forces k key ranges wherever the partial slots allow).
float combine_cost() {
  static const float c = [] {
    const char* e = std::getenv("SPECFOLD_ATTN_COMBINE_COST");
    return e ? static_cast<float>(std::atof(e)) : 8.f;
  }();
  return c;
}

template <int HD>
int run_attn(const AttnCall& c, cudaStream_t st) {
  using C = ACfg<HD>;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  const int R = c.B * c.L;
  const int g = c.n_q / c.n_kv;
  int rc = make_map_2d(&p.mapQ, c.Q, static_cast<uint64_t>(c.n_kv) * R * g, HD, HD, 128);
  if (rc) return rc;
  if (c.P > 0) {
    // contiguous: the map spans the P prefix tokens; paged: the whole pool
    const uint64_t tokens = c.pk.block_table ? static_cast<uint64_t>(c.pk.num_pages) * c.pk.page_size : c.P;
    const uint64_t vtokens = c.pv.block_table ? static_cast<uint64_t>(c.pv.num_pages) * c.pv.page_size : c.P;
    // K in 64-token boxes (the kernel stores a block's K half by half)
    rc = make_map_3d(&p.mapK, c.pk.ptr, HD, c.n_kv, tokens, c.pk.head_stride, c.pk.token_stride, 64);
    if (rc) return rc;
    rc = make_map_3d(&p.mapV, c.pv.ptr, HD, c.n_kv, vtokens, c.pv.head_stride, c.pv.token_stride, 128);
    if (rc) return rc;
    if (c.pk.block_table) {
      p.table = c.pk.block_table;
      p.page_size = c.pk.page_size;
      p.num_pages = std::min(c.pk.num_pages, c.pv.num_pages);
      p.page_tma = c.pk.page_size % 128 == 0 ? 1 : 0;
    }
    p.pkp = static_cast<const __nv_bfloat16*>(c.pk.ptr);
    p.pvp = static_cast<const __nv_bfloat16*>(c.pv.ptr);
    p.k_ts = c.pk.token_stride;
    p.k_hs = c.pk.head_stride;
    p.v_ts = c.pv.token_stride;
    p.v_hs = c.pv.head_stride;
  }
  p.bK = static_cast<const __nv_bfloat16*>(c.blockK);
  p.bV = static_cast<const __nv_bfloat16*>(c.blockV);
  p.src = c.src;
  p.packed_idx = c.packed_idx;
  p.n_dev = c.n_dev;
  p.O = static_cast<__nv_bfloat16*>(c.O);
  p.P = c.P;
  p.L = c.L;
  p.R = R;
  p.n_kv = c.n_kv;
  p.g = g;
  p.n_q = c.n_q;
  p.sl2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(HD)));
  p.status = c.status;
  p.n_early = c.n_early ? 1 : 0;
  p.num_sms = num_sms();
  // split counts per live tile count, within the partials' slot capacity
  const int cap = attn_slot_cap(R, g, c.n_kv);
  const int tiles_max = std::min(((R * g + 127) / 128) * c.n_kv, kSpTable);  // n <= R
  int units_max = ((R * g + 127) / 128) * c.n_kv;  // every tile, unsplit
  bool any_split = false;
  static const int forced_sp = env_int("SPECFOLD_ATTN_SPLITS", 0);  // > 0: that split count wherever it fits
  for (int t = 1; t <= tiles_max; ++t) {
    const int lim = std::min(16, cap / t);
    int sp = lim >= 2 ? plan_splits(t, lim, p.num_sms, c.P, combine_cost()) : 1;
    if (forced_sp > 0) sp = std::max(1, std::min(forced_sp, std::max(lim, 1)));
    p.sp_table[t - 1] = static_cast<uint8_t>(sp);
    units_max = std::max(units_max, t * sp);
    any_split = any_split || sp > 1;
  }
  if (cap > 0) {
    if (!c.part || c.part_bytes < attn_partial_bytes(R, g, c.n_kv, HD)) return SPECFOLD_ECAPACITY;
    p.part_o = static_cast<float*>(c.part);
    p.part_ml = p.part_o + static_cast<size_t>(cap) * 128 * HD;
  }
  if (const int rc = smem_limit_once(attn_kernel<HD>, C::SMEM_BYTES)) return rc;
  // FFN weight prefetch by CTAs without a unit: the leading k-blocks of the
  // gate and up weights, about 40 MB (well inside L2 next to the output
  // projection's weights and the layer's activations)
  static const int pf_wo = env_int("SPECFOLD_PREFETCH_WO", 0);
  static const int pf_ffn_mb = env_int("SPECFOLD_FFN_PREFETCH_MB", 40);
  static const int pf_pace = env_int("SPECFOLD_PREFETCH_PACE_NS", 400);
  static const int pf_blk = env_int("SPECFOLD_PREFETCH_BLOCK_NS", 1500);
  static const int pf_delay = env_int("SPECFOLD_PREFETCH_DELAY_NS", 3000);
  p.pf_delay_ns = std::min(std::max(pf_delay, 0), 1000000);
  p.pf_pace_ns = std::max(pf_pace, 0);
  p.pf_blk_ns = std::max(pf_blk, 0);
  if (pf_wo && c.wo && c.wo_rows % 128 == 0 && c.wo_cols % 64 == 0 && ffn_prefetch_enabled() &&
      make_map_2d(&p.pf_omap, c.wo, c.wo_rows, c.wo_cols, c.wo_cols, 128) == SPECFOLD_OK) {
    p.pf_orb = c.wo_rows / 128;
    p.pf_okb = c.wo_cols / 64;
  }
  if (c.ffn_w[0] && c.ffn_w[1] && c.ffn_F % 128 == 0 && c.ffn_d % 64 == 0 && ffn_prefetch_enabled()) {
    bool ok = true;
    for (int m = 0; m < 2; ++m)
      ok = ok && make_map_2d(&p.pf_map[m], c.ffn_w[m], c.ffn_F, c.ffn_d, c.ffn_d, 128) == SPECFOLD_OK;
    if (ok) {
      p.pf_n = 2;
      p.pf_rb = c.ffn_F / 128;
      const long long box_bytes = 128LL * 64 * 2;
      p.pf_kb = static_cast<int>(
          std::min<long long>(c.ffn_d / 64, (static_cast<long long>(std::max(pf_ffn_mb, 0)) << 20) / (2LL * p.pf_rb * box_bytes)));
      if (p.pf_kb <= 0) p.pf_n = 0;
    }
  }
  // persistent: at most one CTA per SM, each looping over the live units
  // (every SM when CTAs without a unit have weights to prefetch)
  const dim3 grid(p.pf_n > 0 || p.pf_orb > 0 ? p.num_sms : std::min(units_max, p.num_sms));
  launch_k(attn_kernel<HD>, dim3(grid), dim3(kAttnThreads), C::SMEM_BYTES, st, p);
  count_launch();
  if (check_launch()) return SPECFOLD_ECUDA;
  if (any_split) {  // no combine launch when no row count splits the key range
    const long long work = static_cast<long long>(R) * g * c.n_kv * (HD / 8);
    const int cg = static_cast<int>(std::min<long long>((work + 255) / 256, 8LL * num_sms()));
    launch_k(attn_combine_kernel<HD>, dim3(std::max(cg, 1)), dim3(256), 0, st, p);
    count_launch();
    return check_launch();
  }
  return SPECFOLD_OK;
}

}  // namespace

// Partial slots of the split-KV path: enough for four waves of units on the
// SMs the split sizing plans for, and at most 16 splits of every (query tile,
// KV head) of R rows.  0 when no split is possible.
int attn_slot_cap(int R, int g, int n_kv) {
  const int tiles = ((R * g + 127) / 128) * n_kv;
  const int cap = std::min(16 * tiles, 4 * kSmBudget);
  return cap >= 2 ? cap : 0;
}

size_t attn_partial_bytes(int R, int g, int n_kv, int hd) {
  return static_cast<size_t>(attn_slot_cap(R, g, n_kv)) * 128 * (hd + 2) * sizeof(float);
}

int launch_attention(const AttnCall& c, cudaStream_t st) {
  if (c.hd == 128) return run_attn<128>(c, st);
  if (c.hd == 64) return run_attn<64>(c, st);
  return SPECFOLD_EUNSUPPORTED;
}

}  // namespace sf
