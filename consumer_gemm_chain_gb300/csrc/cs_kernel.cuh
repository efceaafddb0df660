// Persistent tile-synchronised GEMM-chain kernel for sm_103a.
//
// CTAs (or clusters) pull work units from a dependency-ordered schedule
// through a global atomic counter (a megakernel-style task queue: a dependent
// task starts once the slice it reads is done, not when the whole producer op
// is done).  Roles inside a CTA (224 threads; 352 in the attention
// instantiations, which have eight epilogue warps):
//   last warp   : scheduler (warp 6, or 10).  Claims the next unit just in time (when the TMA
//                 warp is a few K-slices from the end of its current unit),
//                 and for consumer units polls the producer tile semaphores of
//                 the unit's K range with all 32 lanes at once, publishing how
//                 many leading producer tiles are complete in shared memory
//                 (acquire at gpu scope, release at CTA scope).
//   warp 0      : TMA producer (lane 0).  Before loading a K-slice of the
//                 intermediate it checks the published readiness (a compare in
//                 the loop, an out-of-line wait at the bound) and fences the
//                 async proxy.
//   warp 1      : TMEM allocator (whole warp) and tcgen05.mma issuer (lane 0).
//   warps 2..5  : epilogue (2..9 for attention: two warps per TMEM lane
//                 quadrant, each on half of a tile's columns): tcgen05.ld of
//                 the fp32 accumulator, bias + GeLU / SiLU*up / none,
//                 downcast, swizzled smem staging, TMA store, then (producer
//                 stages) release-increment of the tile semaphore and of the
//                 row counter; the last K-split of a small tile sums the
//                 splits' partials first.  Attention units run their softmax
//                 here, between the S = QK^T and P V MMAs.
// CG = 2 (pair mode): a 2-CTA cluster shares one 256 x 256 tile.  Each CTA
// loads its 128 rows of A and its half of B's columns; the leader (rank 0)
// issues tcgen05.mma.cta_group::2, whose accumulator rows 0-127 land in the
// leader's TMEM and rows 128-255 in the peer's; commits are multicast to both.
// CL = 4: two such pairs on consecutive 256-row blocks form a 4-CTA cluster
// and share every weight box by TMA multicast.  Attention on pairs runs two
// query blocks per unit.  AR = 8: up to 8 rows, one 8-row A group per stage;
// AR = 32: up to 32 rows, four groups.
// Semaphores stay per 128-row block, so each CTA of a consumer cluster waits
// only for the producer rows it reads.
// Every wait is bounded: semaphore polls by the plan's timeout (error word +
// global abort flag), mbarrier waits by a watchdog (error word + CTA abort).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cs_ptx.cuh"

namespace cs {

constexpr int BM = 128;           // tile rows per CTA (UMMA M per SM)
constexpr int BK = 64;            // K-slice per pipeline stage (128 bytes of fp16/bf16)
constexpr int UMMA_K = 16;        // K per tcgen05.mma (kind::f16)
constexpr int TILE_A_BYTES = BM * BK * 2;  // 16 KB
constexpr int STAGING_BYTES = 2 * BM * 128;  // two 64-column chunk buffers of 128 rows
constexpr int UQ = 4;             // unit-queue depth (scheduler -> TMA/MMA/epilogue)
// Warp roles: 0 TMA, 1 MMA, EPI_WARP0 .. EPI_WARP0 + EPI - 1 epilogue, then the
// scheduler.  Epilogue warp w reads TMEM lane quadrant w % 4; the attention
// instantiations run two epilogue warps per quadrant, each on half of a tile's
// columns (the softmax of a 128-key block is then split over two warps).
constexpr int EPI_WARP0 = 2;
template <bool ATTN>
struct Roles {
  static constexpr int EPI = ATTN ? 8 : 4;
  static constexpr int SCHED = EPI_WARP0 + EPI;
  static constexpr int THREADS = (SCHED + 1) * 32;
};
constexpr int CLAIM_AHEAD = 12;   // K-slices before a unit's end at which the next unit is claimed
constexpr uint32_t READY_ALL = 0x7FFFFFFFu;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t UNIT_END = 0xFFFFFFFFu;

// Control block words (device memory owned by the plan).
enum : int {
  CTRL_DISPATCH = 0,
  CTRL_EXIT = 1,
  CTRL_EPOCH = 2,
  CTRL_ERROR = 3,
  CTRL_ABORT = 4,
  CTRL_ERR_UNIT = 5,
  CTRL_ERR_WHERE = 6,
  CTRL_ERR_CTA = 7,
  CTRL_WORDS = 16
};
enum : uint32_t { ERR_TIMEOUT = 4, ERR_WATCHDOG = 6 };  // == cs_status values

enum : int { STAGE_GEMM = 0, STAGE_ATTN = 1 };
enum : int { EPI_NONE = 0, EPI_BIAS_GELU = 1, EPI_SWIGLU = 2 };
enum : int { WAIT_NONE = 0, WAIT_TILE = 1, WAIT_ROW = 2, WAIT_STRIDED = 3 };

struct StageP {
  int kind;        // STAGE_GEMM / STAGE_ATTN
  int epi;         // EPI_*
  int m_tiles, n_tiles;  // n_tiles: column tiles; semaphores are [128-row blocks][n_tiles]
  int k_iters;     // BK-slices of the reduction
  int n_extent;    // valid output columns (bias guard, store guard)
  int m_extent;    // valid output rows (store guard)
  int bn;          // output columns per tile (128 or 256)
  int mma_n;       // UMMA N (bn, or 256 for gate|up with bn = 128)
  int b_major;     // 0: weights K-major ([N,K]); 1: MN-major ([K,N])
  int map_a, map_b, map_b2, map_out;
  int map_k;  // attention on a CTA pair: QKV loads of 64-row boxes (half a key block)
  void* out_ptr;   // the output (row-major, out_ld elements per row) for plain stores, or null
  long long out_ld;
  int b_bytes;     // bytes of the B operand per pipeline stage and CTA
  const __nv_bfloat16* bias_bf16;  // exactly one of these two is used (per dtype)
  const __half* bias_f16;
  // consumer side
  int wait;        // WAIT_*
  const uint32_t* dep_tile;  // producer tile semaphores [128-row blocks][dep_ntiles]
  const uint32_t* dep_row;   // producer row counters [128-row blocks]
  int dep_ntiles;
  int dep_bn;      // intermediate columns per producer tile
  int stride;      // WAIT_STRIDED stride (producer column tiles)
  // producer side
  uint32_t* rel_tile;  // this stage's tile semaphores (null: no release)
  uint32_t* rel_row;
  const uint32_t* delay_ns;  // per 128-row block x column tile, or null
  int skip_unit;   // 128-row block x column tile that skips its release (-1: none)
  // split-K: `splits` units per tile, each over `kps` K-slices, writing fp32
  // partial tiles [splits][m_blocks][n_tiles][128][mma_n]; the last to arrive
  // (per-tile counter, `splits` arrivals per forward) reduces them in split order
  int splits, kps, m_blocks;
  float* partial;
  uint32_t* split_ctr;
  // Stream-K tail (the last GEMM stage only): the stage's last sk_tiles tiles
  // in dispatch order are replaced by sk_units units that each cover sk_q
  // consecutive K-slices of the tiles' concatenated K ranges (crossing tile
  // boundaries); a tile's contributors write fp32 partials
  // [sk_tiles][sk_max_nc][CTAs per unit][128][mma_n] and count their arrival
  // on split_ctr; the last to arrive sums them in K order, runs the epilogue
  // and releases.  sk_tile[j] is the unit encoding of tile j.
  int sk_tiles, sk_units, sk_q, sk_max_nc;
  float* sk_partial;
  const uint32_t* sk_tile;
  // L2 prefetch of upcoming K-slices by the scheduler warp (null: none):
  // pf_b/pf_b2 = weight base(s), pf_ldb = bytes between weight rows, pf_brows =
  // weight rows (N if K-major, K if MN-major); pf_a/pf_lda/pf_arows likewise for A.
  const char* pf_b;
  const char* pf_b2;
  long long pf_ldb;
  int pf_brows;
  const char* pf_a;
  long long pf_lda;
  int pf_arows;
  // attention (STAGE_ATTN)
  // kv_chunk > 0: the units of tile row m run as ceil((m + 1) / kv_chunk)
  // pieces of at most kv_chunk key groups (CTAs-per-unit key blocks each); a
  // piece writes its fp32 state [query block][head][piece][ATT_PART_COLS][128]
  // to `partial` and counts its arrival on split_ctr[query block * heads + head]
  int kv_chunk, kv_max;
  int heads;
  float softmax_scale_log2;  // log2(e) / sqrt(head_dim)
};

struct KParams {
  CUtensorMap maps[9];
  StageP st[3];
  const uint32_t* sched;
  int n_units;
  uint32_t* ctrl;
  unsigned long long timeout_ns;
  unsigned long long watchdog_ns;
  int bf16;
  int waits;       // consumers wait on semaphores
  int release;     // producers release semaphores
  int bump_epoch;  // this launch completes a forward
  int acc_stride;  // TMEM columns between the two accumulator buffers
  unsigned long long* trace;  // optional per-unit timestamps (TRACE_WORDS per record), or null
  int trace_records;
  int pf_dist;     // L2 prefetch distance in K-slices (0: off)
};

// Trace record of one unit on one CTA (index = dispatch index * CTAs per tile + rank):
//   [0] unit | dispatch index << 32   [1] smid | blockIdx << 16 | rank << 30
//   [2] claimed   [3] dependencies published   [4] first TMA load   [5] last TMA load
//   [6] accumulator complete (epilogue)   [7] epilogue done (stores + release)
constexpr int TRACE_WORDS = 8;
__device__ __forceinline__ uint32_t smid() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void trace_put(const KParams& p, uint32_t idx, uint32_t rank, int cg, int word,
                                          unsigned long long v) {
  if (p.trace == nullptr) return;
  const uint32_t rec = idx * static_cast<uint32_t>(cg) + rank;
  if (rec < static_cast<uint32_t>(p.trace_records)) p.trace[static_cast<size_t>(rec) * TRACE_WORDS + word] = v;
}

template <int NS>
struct SmemCtl {
  uint64_t full[NS], empty[NS];
  uint64_t tfull[2], tempty[2];
  uint64_t uq_full[UQ], uq_empty[UQ];
  uint64_t s_full, p_full, o_full;  // attention: S ready, P written, O_j ready
  uint64_t s_full_b;  // pair attention: S of odd key blocks (its own phases)
  uint64_t drain;
  uint64_t claim_req;       // TMA warp -> scheduler: claim the next unit now
  uint64_t mb_full, mb_empty;  // pair mode: leader -> peer unit mailbox
  uint32_t uq[UQ];
  uint32_t uq_idx[UQ];      // dispatch index of each queued unit (trace records)
  uint32_t uq_ready[UQ];    // per queued unit: leading producer items known complete
  uint32_t uq_kb[UQ];       // per queued piece: first K-slice | end K-slice << 16
  uint32_t uq_part[UQ];     // per queued piece: contributor | contributors << 8 | last of its claim << 15 |
                            // Stream-K tile << 16 (0xFFFF: a tile unit)
  uint32_t mb_unit;         // pair mode: dispatch index handed to the peer
  uint32_t tmem_base;
  volatile int abort;
  volatile int split_last;  // epilogue: this unit was the last split of its tile
  volatile int tma_seq;     // TMA warp: units started so far
  volatile int tma_kb;      // TMA warp: K-slice of its latest load
  int issued_parity[NS];  // TMA thread: parity of the last load issued into each slot (-1: none)
  uint4 bias_s[32];       // epilogue: the bias of one tile (up to 256 values)
  float xchg[2][BM];      // attention epilogue: the two warps of a row exchange row maxima and sums
};

__device__ __forceinline__ void record_error(const KParams& p, uint32_t code, uint32_t unit, uint32_t where) {
  if (atomicCAS(&p.ctrl[CTRL_ERROR], 0u, code) == 0u) {
    p.ctrl[CTRL_ERR_UNIT] = unit;
    p.ctrl[CTRL_ERR_WHERE] = where;
    p.ctrl[CTRL_ERR_CTA] = blockIdx.x;
  }
  atomicExch(&p.ctrl[CTRL_ABORT], 1u);
  __threadfence();
}

// Bounded mbarrier wait.  False when the CTA is aborting or the watchdog fired.
// CLUSTER: acquire at cluster scope (the arrivals come from the peer CTA).
template <int NS, bool CLUSTER = false>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, SmemCtl<NS>* sc, const KParams& p,
                                         uint32_t where) {
  auto try_once = [&]() { return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (try_once()) return true;
  const uint64_t t0 = globaltimer();
  uint32_t it = 0;
  while (true) {
    if (try_once()) return true;
    if (sc->abort) return false;
    if ((++it & 63u) == 0u && globaltimer() - t0 > p.watchdog_ns) {
      record_error(p, ERR_WATCHDOG, 0xFFFFFFFFu, where);
      sc->abort = 1;
      return false;
    }
  }
}

// Unit encoding: stage [31:30] | K-split [29:26] | tile row [25:14] | tile column [13:0].
__device__ __forceinline__ uint32_t unit_stage(uint32_t u) { return u >> 30; }
__device__ __forceinline__ int unit_ks(uint32_t u) { return static_cast<int>((u >> 26) & 0xFu); }
__device__ __forceinline__ int unit_m(uint32_t u) { return static_cast<int>((u >> 14) & 0xFFFu); }
__device__ __forceinline__ int unit_n(uint32_t u) { return static_cast<int>(u & 0x3FFFu); }
// A schedule entry with K-split field SK_KS is Stream-K unit unit_n(u) of its stage.
constexpr int SK_KS = 15;

// A queued piece of work: a tile unit, or one tile's share of a Stream-K unit.
__device__ __forceinline__ int piece_kb0(uint32_t kb) { return static_cast<int>(kb & 0xFFFFu); }
__device__ __forceinline__ int piece_kb1(uint32_t kb) { return static_cast<int>(kb >> 16); }
__device__ __forceinline__ int part_c(uint32_t x) { return static_cast<int>(x & 0xFFu); }
__device__ __forceinline__ int part_nc(uint32_t x) { return static_cast<int>((x >> 8) & 0x7Fu); }
__device__ __forceinline__ bool part_last(uint32_t x) { return ((x >> 15) & 1u) != 0u; }
__device__ __forceinline__ int part_sk(uint32_t x) { return static_cast<int>(x >> 16); }
constexpr uint32_t PART_TILE = 0xFFFFu << 16;  // not a Stream-K tile
constexpr uint32_t PART_LAST = 1u << 15;

struct RingPos {
  uint32_t slot = 0, phase = 0;
  template <int NS>
  __device__ __forceinline__ void next() {
    if (++slot == NS) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Scheduler warp: poll the producer flags a consumer unit depends on and
// publish, in sc->uq_ready[q], how many leading dependency items are complete.
// Items are producer column tiles 0..dep_ntiles-1 of 128-row block m, in the
// order the consumer's K-loop reads them: TILE publishes the first incomplete
// tile of the unit's own K range (the tiles before that range count as
// complete: a K-split reads none of them); ROW publishes 0 until the row
// counter is complete, then dep_ntiles; STRIDED publishes the smallest residue
// class (mod stride) with an incomplete tile.  Flags are read with relaxed
// loads (32 lanes in parallel) and each observing lane fences (acquire
// pattern) before the CTA-scope release.
template <int NS>
__device__ void sched_poll_gemm(const KParams& p, const StageP& S, SmemCtl<NS>* sc, uint32_t q, int m,
                                uint32_t epoch1, uint32_t unit, int kb0, int kb1, int lane) {
  const uint32_t* tiles = S.dep_tile + static_cast<size_t>(m) * S.dep_ntiles;
  // TILE: the unit reads producer tiles [i0, i1)
  const int i0 = S.wait == WAIT_TILE ? (kb0 * BK) / S.dep_bn : 0;
  const int nt = S.wait == WAIT_TILE ? min(S.dep_ntiles, ((kb1 - 1) * BK) / S.dep_bn + 1) : S.dep_ntiles;
  int published = 0;
  const uint64_t t0 = globaltimer();
  uint32_t ns = 64;
  while (true) {
    int ready;
    if (S.wait == WAIT_ROW) {
      uint32_t v = lane == 0 ? ld_relaxed_gpu(S.dep_row + m) : 0u;
      v = __shfl_sync(0xFFFFFFFFu, v, 0);
      ready = static_cast<int32_t>(v - epoch1 * static_cast<uint32_t>(nt)) >= 0 ? nt : 0;
    } else {
      ready = nt;
      for (int base = i0; base < nt; base += 32) {
        const int t = base + lane;
        const bool done = t >= nt || static_cast<int32_t>(ld_relaxed_gpu(tiles + t) - epoch1) >= 0;
        const uint32_t bad = __ballot_sync(0xFFFFFFFFu, !done);
        if (S.wait == WAIT_TILE) {
          if (bad) {
            ready = base + __ffs(bad) - 1;
            break;
          }
        } else {  // STRIDED: residue class of each incomplete tile
          int mn = done ? 0x7FFFFFFF : (t % S.stride);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
          if (mn < ready) ready = mn;
        }
      }
    }
    if (ready > published) {
      fence_acq_rel_gpu();
      __syncwarp();
      if (lane == 0) st_release_cta_shared(&sc->uq_ready[q], static_cast<uint32_t>(ready));
      published = ready;
    }
    if (published >= nt) return;
    bool give_up = false;
    if (lane == 0) {
      if (ld_relaxed_gpu(&p.ctrl[CTRL_ABORT]) != 0u) {
        give_up = true;
      } else if (globaltimer() - t0 > p.timeout_ns) {
        record_error(p, ERR_TIMEOUT, unit, static_cast<uint32_t>(published));
        give_up = true;
      }
    }
    give_up = __shfl_sync(0xFFFFFFFFu, give_up ? 1 : 0, 0) != 0;
    if (give_up) {
      // the forward is void; let the pipeline drain without the data
      if (lane == 0) st_release_cta_shared(&sc->uq_ready[q], READY_ALL);
      return;
    }
    __nanosleep(ns);
    if (ns < 512) ns <<= 1;
  }
}

// TMA thread: wait until the scheduler has published at least `need` items
// for queue slot q (shared memory only), then fence the async proxy so the
// TMA loads that follow see the intermediate the producers stored.
template <int NS>
__device__ __forceinline__ bool tma_wait_ready(SmemCtl<NS>* sc, uint32_t q, int need, int& cached,
                                               const KParams& p) {
  if (cached >= need) return true;
  const uint64_t t0 = globaltimer();
  uint32_t it = 0;
  while (true) {
    const int v = static_cast<int>(ld_acquire_cta_shared(&sc->uq_ready[q]));
    if (v >= need) {
      cached = v;
      fence_proxy_async_global();
      return true;
    }
    if (sc->abort) return false;
    if ((++it & 63u) == 0u && globaltimer() - t0 > p.watchdog_ns) {
      record_error(p, ERR_WATCHDOG, 0xFFFFFFFFu, 8);
      sc->abort = 1;
      return false;
    }
    __nanosleep(32);
  }
}

// TMA thread, out of line: wait until slice kb of a consumer unit may load
// (the scheduler has published at least kb * BK / dep_bn + 1 complete
// producer tiles) and return the first slice that is not yet known to be
// loadable, or -1 after an abort or a watchdog timeout.  Kept out of the K
// loop so that the loop itself carries only one integer compare.
template <int NS>
__device__ __noinline__ int tma_wait_slices(SmemCtl<NS>* sc, uint32_t q, int kb, int dep_bn, const KParams& p) {
  int ready = 0;
  if (!tma_wait_ready(sc, q, (kb * BK) / dep_bn + 1, ready, p)) return -1;
  const long long lim = (static_cast<long long>(ready) * dep_bn + BK - 1) / BK;
  return lim > 0x7FFFFFFFLL ? 0x7FFFFFFF : static_cast<int>(lim);
}

// ---------------------------------------------------------------- TMA role
// CL = CTAs per unit: 1, 2 (a pair sharing one 256-row MMA) or 4 (two pairs
// on consecutive 256-row blocks of the same column tile: each weight box is
// fetched once and multicast to the CTA holding the same B columns in the
// other pair).
// AR: A rows held in shared memory per stage: 128, 8 for up to 8 valid rows
// (the MMA then reads the one 8-row group for every 8-row group of its 128
// rows) or 32 for up to 32 (its rows 32-127 read the stage's B operand); the
// accumulator rows past the valid ones are never stored.
template <int NS, int STAGE_BYTES, int CG, int CL, int AR>
__device__ bool tma_gemm_unit(const KParams& p, SmemCtl<NS>* sc, uint8_t* ring, RingPos& rp, uint32_t unit,
                              uint32_t q, uint32_t rank) {
  const uint32_t tidx = sc->uq_idx[q];
  const StageP& S = p.st[unit_stage(unit)];
  const int m = unit_m(unit), n = unit_n(unit);
  constexpr int A_BYTES = AR * BK * 2;
  const uint32_t bytes = A_BYTES + S.b_bytes;
  const bool do_wait = p.waits && S.wait != WAIT_NONE;
  const int kb0 = piece_kb0(sc->uq_kb[q]);
  const int kb1 = piece_kb1(sc->uq_kb[q]);
  // the next unit is claimed near the end of the last piece of this claim
  const int claim_at = !part_last(sc->uq_part[q]) ? -1 : kb1 - kb0 > CLAIM_AHEAD ? kb1 - CLAIM_AHEAD : kb0;
  const int row0 = (m * CL + static_cast<int>(rank)) * BM;  // this CTA's A rows
  const int prank = static_cast<int>(rank) & (CG - 1);        // rank inside the MMA pair
  // gate|up on a pair: the MMA's N = 2*bn is split over the two CTAs, so the
  // first holds the bn gate rows of B and the second the bn up rows
  const bool gate_up = CG == 2 && S.map_b2 >= 0;
  const int bcols = gate_up ? S.bn : S.bn / CG;              // this CTA's share of B's rows
  const int col0 = n * S.bn + (gate_up ? 0 : prank * bcols);
  const int map_b = gate_up && prank == 1 ? S.map_b2 : S.map_b;
  // activations and the intermediate stay in L2, the weights stream through
  const uint64_t pol_a = policy_evict_last();
  const uint64_t pol_b = policy_evict_first();
  int ready_kb = do_wait ? kb0 : kb1;  // slices below this bound may load now
  for (int kb = kb0; kb < kb1; ++kb) {
    if (rank == 0 && kb == claim_at) mbar_arrive(&sc->claim_req);
    if (kb >= ready_kb) {
      ready_kb = tma_wait_slices(sc, q, kb, S.dep_bn, p);
      if (ready_kb < 0) return false;
    }
    if (!wait_bar(&sc->empty[rp.slot], rp.phase ^ 1u, sc, p, 1)) return false;
    uint8_t* sa = ring + rp.slot * STAGE_BYTES;
    uint8_t* sb = sa + A_BYTES;
    // Completion goes to the pair leader's full barrier: each CTA of a pair adds
    // its bytes (with CL = 4 its A, and its B columns: one half fetched here,
    // one multicast by the other pair, which counts them on this pair's leader).
    uint32_t bar_addr;
    if constexpr (CG == 1) {
      bar_addr = smem_u32(&sc->full[rp.slot]);
      mbar_arrive_expect_tx(&sc->full[rp.slot], bytes);
    } else {
      bar_addr = mapa_shared(&sc->full[rp.slot], rank & ~1u);
      if ((rank & 1u) == 0u)
        mbar_arrive_expect_tx(&sc->full[rp.slot], bytes);
      else
        mbar_expect_tx_remote(bar_addr, bytes);
    }
    auto load = [&](void* dst, const CUtensorMap* map, int x, int y, uint64_t pol) {
      if constexpr (CG == 1)
        tma_load_2d_h(dst, map, x, y, &sc->full[rp.slot], pol);
      else
        tma_load_2d_pair_h(dst, map, x, y, bar_addr, pol);
    };
    if (kb == kb0) {
      sc->tma_seq = sc->tma_seq + 1;
      trace_put(p, tidx, rank, CL, 4, globaltimer());
    }
    sc->tma_kb = kb;
    if (kb == kb1 - 1) trace_put(p, tidx, rank, CL, 5, globaltimer());
    load(sa, &p.maps[S.map_a], kb * BK, row0, pol_a);
#ifndef CS_NO_CLUSTER_MULTICAST
    if constexpr (CL == 4) {
      // this CTA fetches half of its B columns (the half of its pair index)
      // for itself and for the CTA with the same pair rank in the other pair
      const uint16_t mask = static_cast<uint16_t>((1u << prank) | (1u << (prank + 2)));
      const int part = static_cast<int>(rank) >> 1;
      const CUtensorMap* bm = &p.maps[map_b];
      if (S.b_major == 0) {
        // weights [N, K]: a box of 64 K x bcols/2 N rows
        tma_load_2d_mc_pair_h(sb + part * (bcols / 2) * (BK * 2), bm, kb * BK, col0 + part * (bcols / 2), bar_addr,
                              mask, pol_b);
      } else {
        // weights [K, N]: every other 64-column box (8 KB each)
        for (int h = part; h < bcols / 64; h += 2)
          tma_load_2d_mc_pair_h(sb + h * 8192, bm, col0 + h * 64, kb * BK, bar_addr, mask, pol_b);
      }
      sc->issued_parity[rp.slot] = static_cast<int>(rp.phase);
      rp.next<NS>();
      continue;
    }
#endif  // CS_NO_CLUSTER_MULTICAST
    // B operand(s): this CTA's bcols rows of N per operand; a second operand
    // (the up projection of gate|up) follows the first, so one N = 2*bn MMA
    // covers both.
    const int nops = S.map_b2 >= 0 && !gate_up ? 2 : 1;
    for (int op = 0; op < nops; ++op) {
      const CUtensorMap* bm = &p.maps[op == 0 ? map_b : S.map_b2];
      uint8_t* dst = sb + op * bcols * (BK * 2);
      if (S.b_major == 0) {
        // weights [N, K]: one box of 64 K x bcols N rows
        load(dst, bm, kb * BK, col0, pol_b);
      } else {
        // weights [K, N]: boxes of 64 N (contiguous) x 64 K rows (8 KB), one per 64 columns
        for (int h = 0; h < bcols / 64; ++h) load(dst + h * 8192, bm, col0 + h * 64, kb * BK, pol_b);
      }
    }
    sc->issued_parity[rp.slot] = static_cast<int>(rp.phase);
    rp.next<NS>();
  }
  return true;
}

// ---------------------------------------------------------------- MMA role
template <int NS, int STAGE_BYTES, int CG, int CL, int AR>
__device__ bool mma_gemm_unit(const KParams& p, SmemCtl<NS>* sc, uint8_t* ring, RingPos& rp, uint32_t unit,
                              int kb0, int kb1, uint32_t& acc, uint32_t& acc_phase, uint32_t rank) {
  // a freed stage is refilled by this pair and (CL = 4) by the other pair's
  // multicast: the release goes to every CTA that writes into it
  const uint16_t empty_mask = CL == 4 ? 0xF : 0x3;
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (rank & 2u));
  const StageP& S = p.st[unit_stage(unit)];
  const uint32_t idesc = make_idesc_f16(p.bf16, S.b_major, BM * CG, S.mma_n);
  if (!wait_bar(&sc->tempty[acc], acc_phase ^ 1u, sc, p, 2)) return false;
  tc_fence_after();
  const uint32_t d = sc->tmem_base + acc * static_cast<uint32_t>(p.acc_stride);
  for (int kb = kb0; kb < kb1; ++kb) {
    if (!wait_bar(&sc->full[rp.slot], rp.phase, sc, p, 3)) return false;
    tc_fence_after();
    const uint32_t sa = smem_u32(ring + rp.slot * STAGE_BYTES);
    const uint32_t sb = sa + AR * BK * 2;
    // AR = 8: stride 0 between 8-row groups, so every group reads the one loaded;
    // AR = 32: rows 32-127 run on into the stage's B slice (finite values, rows
    // that are never stored)
    const uint64_t adesc = smem_desc_sw128(sa, 16, AR >= 16 ? 1024 : 0);
    // K-major B: 8-row groups 1024 B apart.  MN-major B: 64-column atoms 8 KB
    // apart (LBO), 8-row K groups 1024 B apart (SBO).
    const uint64_t bdesc = S.b_major == 0 ? smem_desc_sw128(sb, 16, 1024) : smem_desc_sw128(sb, 8192, 1024);
#pragma unroll
    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
      const uint64_t a = adesc + static_cast<uint64_t>(kk * 2);  // +32 bytes along K
      const uint64_t b = bdesc + static_cast<uint64_t>(S.b_major == 0 ? kk * 2 : kk * 128);  // +32 B / +16 rows
      tc_mma_f16<CG>(d, a, b, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
    }
    tc_commit<CG>(&sc->empty[rp.slot], empty_mask);
    rp.next<NS>();
  }
  tc_commit<CG>(&sc->tfull[acc], pair_mask);
  acc ^= 1u;
  if (acc == 0u) acc_phase ^= 1u;
  return true;
}

// ---------------------------------------------------------------- epilogue role
// tanh-form GeLU: x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), with the
// hardware tanh approximation (its error is below the fp16/bf16 rounding of
// the stored intermediate).
__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float k1 = 0.044715f;
  const float u = k0 * x * fmaf(k1 * x, x, 1.0f);
  const float hx = 0.5f * x;
  return fmaf(hx, tanh_approx(u), hx);
}
// SiLU(x) = x * sigmoid(x) = x/2 (1 + tanh(x/2)).
__device__ __forceinline__ float silu_f(float x) {
  const float hx = 0.5f * x;
  return fmaf(hx, tanh_approx(hx), hx);
}

// 64 bias values of columns [col0, col0 + 64) as floats (0 past the end);
// the extent is a multiple of 8, so each 16-byte group is wholly in or out.
__device__ __forceinline__ void load_bias64(const StageP& S, int col0, int bf16, float (&b)[64]) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int col = col0 + g * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (col < S.n_extent)
      v = ldg_nc_v4(bf16 ? static_cast<const void*>(S.bias_bf16 + col) : static_cast<const void*>(S.bias_f16 + col));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f;
      if (bf16)
        f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      else
        f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      b[g * 8 + 2 * i] = f.x;
      b[g * 8 + 2 * i + 1] = f.y;
    }
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b, int bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Write one thread's 64 packed values (32 words) into the 128-byte-swizzled
// staging row `row` of chunk buffer `chunk` (layout expected by a 128B-swizzle
// TMA store and by a K-major SW128 UMMA operand).
__device__ __forceinline__ void stage_row(uint8_t* staging, int chunk, int row, const uint32_t (&w)[32]) {
  uint8_t* base = staging + chunk * (BM * 128) + row * 128;
#pragma unroll
  for (int pc = 0; pc < 8; ++pc) {
    const uint32_t off = static_cast<uint32_t>((pc ^ (row & 7)) << 4);
    const uint32_t addr = smem_u32(base + off);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[pc * 4 + 0]), "r"(w[pc * 4 + 1]),
                 "r"(w[pc * 4 + 2]), "r"(w[pc * 4 + 3])
                 : "memory");
  }
}

// Producer release: all epilogue threads have their stores complete; one thread
// publishes the 128-row block's tile (and its row) with gpu-scope release.
template <int NE>
__device__ void release_tile(const KParams& p, const StageP& S, int mb, int n, int lane) {
  if (lane == 0) {
    tma_store_wait_all<0>();
    fence_proxy_async_global();
  }
  named_bar_sync(1, NE * 32);
  if (threadIdx.x == EPI_WARP0 * 32) {
    const int u = mb * S.n_tiles + n;
    if (S.delay_ns != nullptr) {
      const uint64_t d = S.delay_ns[u] > 10000000u ? 10000000u : S.delay_ns[u];
      if (d) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < d) __nanosleep(256);
      }
    }
    if (p.release && S.rel_tile != nullptr && u != S.skip_unit) {
      // the barrier above ordered every epilogue thread's stores (the TMA
      // stores waited for and fenced to the generic proxy) before this release
      red_release_gpu_add(S.rel_tile + u, 1u);
      red_release_gpu_add(S.rel_row + mb, 1u);
    }
  }
}

// K-split reduction for a row block with few valid rows (R <= 32): the NE * 32
// epilogue threads share the (row, 4-column group) elements of `npc` 64-column
// parts (the value chunks c0 .. c0+nc-1, then for SwiGLU the same up chunks)
// and fetch every split of an element at once; each element is summed in split
// order (the same order as the row-per-thread path, so the same bits) and
// written to the staging buffer as fp32 [part][row][16 float4], the float4 of
// column group g of row r at slot g ^ (r & 15).  EB elements x KSB splits = 16
// loads in flight per thread.  Split ks's tile starts at tile0 + ks * kstride.
template <int EB, int KSB, int NE>
__device__ __forceinline__ void split_reduce_small(const StageP& S, const float4* tile0, size_t kstride, int R,
                                                   int npc, int nc, int c0, float4* sm) {
  const int E = npc * R * 16;
  const int tid = threadIdx.x - EPI_WARP0 * 32;
#pragma unroll 1
  for (int base = tid; base < E; base += NE * 32 * EB) {
    float4 x[EB][KSB];
#pragma unroll
    for (int u = 0; u < EB; ++u) {
      const int e = base + u * NE * 32;
      // element e -> part pc, column group g, row r (rows fastest: coalesced)
      const int pc = e / (R * 16), rem = e - pc * R * 16;
      const int g = rem / R, r = rem - g * R;
      const int col4 = ((pc / nc) * S.bn + (c0 + pc % nc) * 64) / 4 + g;
#pragma unroll
      for (int ks = 0; ks < KSB; ++ks)
        x[u][ks] = (e < E && ks < S.splits) ? __ldcg(tile0 + ks * kstride + col4 * BM + r)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < EB; ++u) {
      const int e = base + u * NE * 32;
      if (e < E) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int ks = 0; ks < KSB; ++ks)
          if (ks < S.splits) s.x += x[u][ks].x, s.y += x[u][ks].y, s.z += x[u][ks].z, s.w += x[u][ks].w;
        const int pc = e / (R * 16), rem = e - pc * R * 16;
        const int g = rem / R, r = rem - g * R;
        sm[(pc * R + r) * 16 + (g ^ (r & 15))] = s;
      }
    }
  }
}

// The last K-split of a tile with at most 32 valid rows: cooperative passes
// bring every split of the tile's 64-column parts (as many per pass as the
// staging buffer holds: all of them up to 32 rows) and, once, the bias on chip;
// each row thread finishes its rows' chunks and writes them with plain 16-byte
// stores, so no staging output, TMA store or per-chunk round trip stays on the
// hand-off to the consumers (measured at GPT-3 M=1: 13 us from accumulator to
// release with the per-chunk path).  With two warps per lane quadrant each
// takes every other chunk of its rows.  The caller fences and releases.
template <int NS, int NE, bool ACT>
__device__ void epi_split_rows_small(const KParams& p, const StageP& S, SmemCtl<NS>* sc, uint8_t* staging,
                                     const float4* tile0, size_t kstride, int R, int mb, int n, int row, int lane) {
  const int nchunks = S.bn / 64;
  const int np = S.epi == EPI_SWIGLU ? 2 : 1;
  // chunks per pass: np parts each, R rows of 256 bytes per part
  const int cap = (STAGING_BYTES / 256) / R / np;
  const int cpp = cap < nchunks ? cap : nchunks;
  // every store still reading the staging buffer is done before it is reused
  if (lane == 0) tma_store_wait_read<0>();
  named_bar_sync(1, NE * 32);
  const int tid = threadIdx.x - EPI_WARP0 * 32;
  constexpr int NH = NE / 4;
  const int half = tid >> 7;  // which of the quadrant's warps
  if (ACT && S.epi == EPI_BIAS_GELU && tid < S.bn / 8) {
    const int col = n * S.bn + tid * 8;  // 16-byte groups, zero past the extent (a multiple of 8)
    uint4 v = make_uint4(0, 0, 0, 0);
    if (col < S.n_extent)
      v = ldg_nc_v4(p.bf16 ? static_cast<const void*>(S.bias_bf16 + col) : static_cast<const void*>(S.bias_f16 + col));
    sc->bias_s[tid] = v;
  }
  float4* sm = reinterpret_cast<float4*>(staging);
  char* out_row = static_cast<char*>(S.out_ptr) + (static_cast<long long>(mb) * BM + row) * S.out_ld * 2;
#pragma unroll 1
  for (int c0 = 0; c0 < nchunks; c0 += cpp) {
    const int nc = nchunks - c0 < cpp ? nchunks - c0 : cpp;
    // the row threads are done with the previous pass's sums
    if (c0 > 0) named_bar_sync(1, NE * 32);
    if (S.splits <= 2)
      split_reduce_small<8, 2, NE>(S, tile0, kstride, R, np * nc, nc, c0, sm);
    else if (S.splits <= 4)
      split_reduce_small<4, 4, NE>(S, tile0, kstride, R, np * nc, nc, c0, sm);
    else if (S.splits <= 8)
      split_reduce_small<2, 8, NE>(S, tile0, kstride, R, np * nc, nc, c0, sm);
    else
      split_reduce_small<1, 16, NE>(S, tile0, kstride, R, np * nc, nc, c0, sm);
    named_bar_sync(1, NE * 32);
    if (row >= R) continue;
#pragma unroll 1
    for (int cc = half; cc < nc; cc += NH) {
      float va[64], vu[64];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 a = sm[(cc * R + row) * 16 + (j ^ (row & 15))];
        va[4 * j] = a.x, va[4 * j + 1] = a.y, va[4 * j + 2] = a.z, va[4 * j + 3] = a.w;
        if (ACT && S.epi == EPI_SWIGLU) {
          const float4 b = sm[((nc + cc) * R + row) * 16 + (j ^ (row & 15))];
          vu[4 * j] = b.x, vu[4 * j + 1] = b.y, vu[4 * j + 2] = b.z, vu[4 * j + 3] = b.w;
        } else {
          vu[4 * j] = vu[4 * j + 1] = vu[4 * j + 2] = vu[4 * j + 3] = 0.0f;
        }
      }
      const int c = c0 + cc;
      uint32_t w[32];
      if (ACT && S.epi == EPI_BIAS_GELU) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 bv = sc->bias_s[c * 8 + g];
          const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2) {
            float2 f;
            if (p.bf16)
              f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[i2]));
            else
              f = __half22float2(*reinterpret_cast<const __half2*>(&bw[i2]));
            const int j = g * 8 + 2 * i2;
            w[j >> 1] = pack2(gelu_tanh_f(va[j] + f.x), gelu_tanh_f(va[j + 1] + f.y), p.bf16);
          }
        }
      } else if (ACT && S.epi == EPI_SWIGLU) {
#pragma unroll
        for (int j = 0; j < 64; j += 2)
          w[j >> 1] = pack2(silu_f(va[j]) * vu[j], silu_f(va[j + 1]) * vu[j + 1], p.bf16);
      } else {
#pragma unroll
        for (int j = 0; j < 64; j += 2) w[j >> 1] = pack2(va[j], va[j + 1], p.bf16);
      }
      const int col0 = n * S.bn + c * 64;
#pragma unroll
      for (int g = 0; g < 8; ++g)
        if (col0 + g * 8 < S.n_extent)
          *reinterpret_cast<uint4*>(out_row + static_cast<long long>(col0 + g * 8) * 2) =
              make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
    }
  }
  // every thread is done reading the sums in the staging buffer before any
  // warp's next unit writes it (attention P, output staging)
  named_bar_sync(1, NE * 32);
}

// NE epilogue warps: with 8, the two warps of a TMEM lane quadrant take every
// other 64-column chunk (and every other 32-column part of a K-split's
// partial).  ACT: the bias + GeLU and SiLU-up epilogues are compiled in (the
// attention instantiations' GEMMs have none).
template <int NS, int CG, int CL, int NE, bool ACT>
__device__ bool epi_gemm_unit(const KParams& p, SmemCtl<NS>* sc, uint8_t* staging, uint32_t unit, uint32_t part,
                              uint32_t& acc, uint32_t& acc_phase, int& last_buf, uint32_t rank, uint32_t tidx,
                              uint32_t epoch1) {
  const StageP& S = p.st[unit_stage(unit)];
  const int mb = unit_m(unit) * CL + static_cast<int>(rank);  // this CTA's 128-row block
  const int n = unit_n(unit);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lane quadrant this warp may access
  const int row = q * 32 + lane;
  constexpr int NH = NE / 4;
  const int half = (warp - EPI_WARP0) >> 2;  // which of the quadrant's warps
  if (!wait_bar(&sc->tfull[acc], acc_phase, sc, p, 4)) return false;
  tc_fence_after();
  if (threadIdx.x == EPI_WARP0 * 32) trace_put(p, tidx, rank, CL, 6, globaltimer());
  const uint32_t tbase =
      sc->tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * static_cast<uint32_t>(p.acc_stride);
  const int nchunks = S.bn / 64;
  // contributors of this tile: its K-splits, or the Stream-K units whose K
  // ranges touch it (this piece is contributor c of nc, in K order)
  const int nc = part_nc(part), skj = part_sk(part);
  const bool split = nc > 1;
  // rows of this block inside the output (the last block may be ragged)
  const int rows_valid = max(0, min(BM, S.m_extent - mb * BM));
  const size_t tile_floats = static_cast<size_t>(BM) * S.mma_n;
  // Partial tiles are stored [mma_n/4][128 rows][4 columns]: the float4 of
  // columns 4c..4c+3 of this thread's row sits at (c * 128 + row), so a warp
  // reads or writes 512 contiguous bytes per access.
  // the row this thread reduces and stores and the lane quadrant of its store
  // box: its own, unless the valid rows are shared out below
  int rrow = row, rq = q;
  auto tile_partial = [&](int ks) {
    if (skj != 0xFFFF)
      return reinterpret_cast<float4*>(
                 S.sk_partial +
                 (static_cast<size_t>(skj * S.sk_max_nc + ks) * CL + rank) * tile_floats) + rrow;
    return reinterpret_cast<float4*>(S.partial + (static_cast<size_t>(ks * S.m_blocks + mb) * S.n_tiles + n) *
                                                     tile_floats) + rrow;
  };
  auto release_tmem = [&]() {
    // this warp is done with the accumulator buffer: hand it back to the MMA
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if constexpr (CG == 1)
        mbar_arrive(&sc->tempty[acc]);
      else
        mbar_arrive_cluster(mapa_shared(&sc->tempty[acc], rank & ~1u));
    }
  };
  if (split) {
    // K-split: write this split's fp32 rows, count the arrival; only the last
    // split of the tile goes on (and reduces every split in split order).
    float4* mine = tile_partial(part_c(part));
    for (int c = half; c < S.mma_n / 32; c += NH) {
      uint32_t v[32];
      tmem_ld32(tbase + c * 32, v);
      tc_wait_ld();
      if (row < rows_valid) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          mine[((c * 32 + j) >> 2) * BM] = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                                      __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
      }
    }
    release_tmem();
    acc ^= 1u;
    if (acc == 0u) acc_phase ^= 1u;
    // the CTA barrier orders every thread's partial stores before the one
    // acq_rel arrival (release: this split's partial; acquire, for the last
    // split: every other split's, read after the next barrier)
    named_bar_sync(1, NE * 32);
    if (threadIdx.x == EPI_WARP0 * 32) {
      const uint32_t old = atom_add_acq_rel_gpu(S.split_ctr + mb * S.n_tiles + n, 1u);
      sc->split_last = (old + 1u == epoch1 * static_cast<uint32_t>(nc)) ? 1 : 0;
    }
    named_bar_sync(1, NE * 32);
    if (!sc->split_last) {
      if (threadIdx.x == EPI_WARP0 * 32) trace_put(p, tidx, rank, CL, 7, globaltimer());
      return true;
    }
  }
  // at most 32 valid rows (the last split of the tile): cooperative passes
  // and plain row stores; the loop below is skipped (33 to 48 rows also ran
  // this way until the row-per-thread sums were shared by all four warps,
  // below: then GPT-3 M=40 71.3 -> 68.5 us, LLaMA M=48 53.0 -> 50.9)
  const bool rows_small = split && skj == 0xFFFF && rows_valid <= 32 && S.out_ptr != nullptr;
  if (rows_small) {
    const size_t kstride = static_cast<size_t>(S.m_blocks) * S.n_tiles * (tile_floats / 4);
    epi_split_rows_small<NS, NE, ACT>(p, S, sc, staging, tile_partial(0) - row, kstride, rows_valid, mb, n, row,
                                      lane);
    last_buf = -1;
  }
  // 33 to 64 valid rows (the last K-split; partial sums come from global memory,
  // so any warp may take any row): the warps of the two empty lane quadrants
  // take every other chunk of the valid rows (measured: GPT-3 M=64 74.0 ->
  // 69.2 us, LLaMA M=64 54.3 -> 50.5).  The staging buffers then change
  // hands between warps: every warp's earlier stores must have read them first,
  // and this unit's stores before the next unit writes them again.
  const bool rows_pair = NH == 1 && split && !rows_small && rows_valid <= 64;
  int c_first = half, c_step = NH;
  if (rows_pair) {
    rrow = (q & 1) * 32 + lane;
    rq = q & 1;
    c_first = q >> 1;
    c_step = 2;
    if (lane == 0) tma_store_wait_read<0>();
    named_bar_sync(1, NE * 32);
  }
#pragma unroll 1
  for (int c = c_first; c < (rows_small ? 0 : nchunks); c += c_step) {
    float va[64], vu[64];
    if (split) {
#pragma unroll
      for (int j = 0; j < 64; ++j) va[j] = vu[j] = 0.0f;
      // sum the splits in split order (the same bits whichever split arrived last);
      // loads of one split are issued together, then added
      for (int ks = 0; ks < nc && rrow < rows_valid; ++ks) {
        const float4* src = tile_partial(ks);
        float4 x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = __ldcg(src + ((c * 64) / 4 + j) * BM);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          va[4 * j] += x[j].x, va[4 * j + 1] += x[j].y, va[4 * j + 2] += x[j].z, va[4 * j + 3] += x[j].w;
        if (ACT && S.epi == EPI_SWIGLU) {
#pragma unroll
          for (int j = 0; j < 16; ++j) x[j] = __ldcg(src + ((S.bn + c * 64) / 4 + j) * BM);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            vu[4 * j] += x[j].x, vu[4 * j + 1] += x[j].y, vu[4 * j + 2] += x[j].z, vu[4 * j + 3] += x[j].w;
        }
      }
    } else {
      uint32_t v[2][32];
      uint32_t u[2][32];
      tmem_ld32(tbase + c * 64, v[0]);
      tmem_ld32(tbase + c * 64 + 32, v[1]);
      if (ACT && S.epi == EPI_SWIGLU) {
        tmem_ld32(tbase + S.bn + c * 64, u[0]);
        tmem_ld32(tbase + S.bn + c * 64 + 32, u[1]);
      }
      tc_wait_ld();
      if (c + NH >= nchunks) release_tmem();  // this warp's last chunk
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        va[j] = __uint_as_float(v[j >> 5][j & 31]);
        vu[j] = (ACT && S.epi == EPI_SWIGLU) ? __uint_as_float(u[j >> 5][j & 31]) : 0.0f;
      }
    }
    uint32_t w[32];
    const int col0 = n * S.bn + c * 64;
    if (ACT && S.epi == EPI_BIAS_GELU) {
      float bias[64];
      load_bias64(S, col0, p.bf16, bias);
#pragma unroll
      for (int j = 0; j < 64; j += 2)
        w[j >> 1] = pack2(gelu_tanh_f(va[j] + bias[j]), gelu_tanh_f(va[j + 1] + bias[j + 1]), p.bf16);
    } else if (ACT && S.epi == EPI_SWIGLU) {
#pragma unroll
      for (int j = 0; j < 64; j += 2)
        w[j >> 1] = pack2(silu_f(va[j]) * vu[j], silu_f(va[j + 1]) * vu[j + 1], p.bf16);
    } else {
#pragma unroll
      for (int j = 0; j < 64; j += 2) w[j >> 1] = pack2(va[j], va[j + 1], p.bf16);
    }
    // Two chunk buffers alternate (with two warps per quadrant each warp keeps
    // one: its chunks all have the same parity).  Every earlier store that read this buffer
    // must be done: if the newest committed store read the other buffer, all
    // but that one group suffice; if it read this buffer, wait for all.
    const int buf = c & 1;
    if (lane == 0) {
      if (last_buf == buf)
        tma_store_wait_read<0>();
      else
        tma_store_wait_read<1>();
    }
    __syncwarp();
    stage_row(staging, buf, rrow, w);
    fence_proxy_async_shared();
    __syncwarp();
    // boxes that start past the tensor's end are skipped, not clipped
    const int grow = mb * BM + rq * 32;
    if (col0 < S.n_extent && grow < S.m_extent) {
      if (lane == 0) {
        tma_store_2d(&p.maps[S.map_out], staging + buf * (BM * 128) + rq * 32 * 128, col0, grow);
        tma_store_commit();
      }
      last_buf = buf;
    }
  }
  if (rows_pair) {
    if (lane == 0) tma_store_wait_read<0>();
    named_bar_sync(1, NE * 32);
    last_buf = -1;
  }
  if (!split) {
    acc ^= 1u;
    if (acc == 0u) acc_phase ^= 1u;
  }
  if (S.rel_tile != nullptr) {
    release_tile<NE>(p, S, mb, n, lane);
    last_buf = -1;
  }
  if (threadIdx.x == EPI_WARP0 * 32) trace_put(p, tidx, rank, CL, 7, globaltimer());
  return true;
}

// ---------------------------------------------------------------- attention unit
// One unit = one 128-query block i of one head h (head_dim 128) of causal
// attention over the QKV intermediate [M, 3F] (columns [Q | K | V], head-major).
// For every key block j <= i (FlashAttention-style online softmax):
//   S = Q_i K_j^T            tcgen05, fp32 in TMEM columns [ATT_S_COL, +128)
//   P = exp2(S*c - m)         epilogue warps (one query row per thread), fp16/bf16
//                             into the staging buffers as a K-major SW128 operand
//   O += P V_j                tcgen05 (V is an MN-major B operand), accumulated in
//                             TMEM [ATT_O_COL, +128) across the unit's key blocks
// P is taken against a reference maximum m that is raised only when a row's
// maximum exceeds it by more than 2^ATT_RESCALE_LOG2 (so P <= 2^8); then O and
// l are rescaled by exp2(m_old - m_new) in TMEM first.  O / l is stored like a
// GEMM tile and the (i, h) semaphore released.
constexpr uint32_t ATT_S_COL = 256;
constexpr uint32_t ATT_O_COL = 384;
// fp32 columns of a piece's state per query row: 128 output dims, max, sum, 2 unused
constexpr int ATT_PART_COLS = 132;
// log2 of the largest P the reference maximum allows before O is rescaled
constexpr float ATT_RESCALE_LOG2 = 8.0f;

// Key blocks [j0, j1) of an attention unit; returns the pieces of its tile
// row.  Tile row i sees key groups 0..i (CG key blocks each); with kv_chunk
// = c, piece k (the unit's K-split field) takes groups [k c, min((k + 1) c, i + 1)).
template <int CG>
__device__ __forceinline__ int attn_keys(const StageP& S, uint32_t unit, int& j0, int& j1) {
  const int i = unit_m(unit);
  if (S.kv_chunk <= 0) {
    j0 = 0;
    j1 = (i + 1) * CG;
    return 1;
  }
  const int c = unit_ks(unit);
  j0 = c * S.kv_chunk * CG;
  j1 = min((c + 1) * S.kv_chunk, i + 1) * CG;
  return (i + S.kv_chunk) / S.kv_chunk;
}

// TMA: three 32 KB slots per key block: [Q dims 0-63 | K_j dims 0-63],
// [Q dims 64-127 | K_j dims 64-127], [V_j dims 0-63 | V_j dims 64-127] (128 rows each).
// CG = 2: a unit is two consecutive query blocks of one head on a CTA pair; each
// CTA loads its own Q rows, half of each K block's 128 keys (the N of Q K^T)
// and half of V's 128 head dimensions (the N of P V); completion goes to the
// pair leader's full barrier as in a pair GEMM.
template <int NS, int STAGE_BYTES, int CG>
__device__ bool tma_attn_unit(const KParams& p, SmemCtl<NS>* sc, uint8_t* ring, RingPos& rp, uint32_t unit,
                              uint32_t q, uint32_t rank) {
  const StageP& S = p.st[unit_stage(unit)];
  const uint32_t tidx = sc->uq_idx[q];
  const int i = unit_m(unit), h = unit_n(unit);
  const int F = S.heads * 128;
  const int qb = i * CG + static_cast<int>(rank);  // this CTA's query block
  int j0, j1;
  attn_keys<CG>(S, unit, j0, j1);
  const int nkb = j1 - j0;                         // key blocks of the unit
  const int nslots = 3 * nkb;
  const int claim_at = nslots > CLAIM_AHEAD ? nslots - CLAIM_AHEAD : 0;
  int ready = 0;
  // every row block up to the unit's query blocks (and so every key block it
  // reads) must be complete first
  if (p.waits && S.wait != WAIT_NONE && !tma_wait_ready(sc, q, (i + 1) * CG, ready, p)) return false;
  const CUtensorMap* m = &p.maps[S.map_a];
  int sidx = 0;
  // CG = 2: the MMA computes S for key block j+1 before P V of block j (two S
  // buffers), so the slots go Q|K of blocks 0 and 1, V_0, Q|K_2, V_1, ...
  for (int step = 0; step < 3 * nkb; ++step, ++sidx) {
    int j, part;
    if constexpr (CG == 1) {
      j = step / 3, part = step % 3;
    } else if (step < 4) {
      j = step >> 1, part = step & 1;  // Q|K of key blocks 0 and 1
    } else {
      const int t = step - 4, jj = t / 3, r3 = t % 3;
      if (jj <= nkb - 3) {
        // V_jj, then Q|K of key block jj + 2
        j = r3 == 0 ? jj : jj + 2;
        part = r3 == 0 ? 2 : r3 - 1;
      } else {
        j = nkb - 2 + r3, part = 2;  // the last two V blocks
      }
    }
    {
      if (rank == 0 && sidx == claim_at) mbar_arrive(&sc->claim_req);
      if (!wait_bar(&sc->empty[rp.slot], rp.phase ^ 1u, sc, p, 1)) return false;
      if (sidx == 0) trace_put(p, tidx, rank, CG, 4, globaltimer());
      if (sidx == nslots - 1) trace_put(p, tidx, rank, CG, 5, globaltimer());
      uint8_t* s0 = ring + rp.slot * STAGE_BYTES;
      const int jb = j0 + j;  // key block
      if constexpr (CG == 1) {
        uint64_t* bar = &sc->full[rp.slot];
        mbar_arrive_expect_tx(bar, 2 * TILE_A_BYTES);
        if (part < 2) {
          tma_load_2d(s0, m, h * 128 + part * 64, qb * BM, bar);                    // Q_i dims chunk
          tma_load_2d(s0 + TILE_A_BYTES, m, F + h * 128 + part * 64, jb * BM, bar);  // K_j dims chunk
        } else {
          tma_load_2d(s0, m, 2 * F + h * 128, jb * BM, bar);                        // V_j dims 0-63
          tma_load_2d(s0 + TILE_A_BYTES, m, 2 * F + h * 128 + 64, jb * BM, bar);     // V_j dims 64-127
        }
      } else {
        const uint32_t bar_addr = mapa_shared(&sc->full[rp.slot], 0);
        const uint32_t bytes = part < 2 ? TILE_A_BYTES + TILE_A_BYTES / 2 : TILE_A_BYTES;
        if (rank == 0)
          mbar_arrive_expect_tx(&sc->full[rp.slot], bytes);
        else
          mbar_expect_tx_remote(bar_addr, bytes);
        if (part < 2) {
          // Q rows of this CTA's query block; keys rank*64 .. +63 of block j
          tma_load_2d_pair(s0, m, h * 128 + part * 64, qb * BM, bar_addr);
          tma_load_2d_pair(s0 + TILE_A_BYTES, &p.maps[S.map_k], F + h * 128 + part * 64, jb * BM + rank * 64,
                           bar_addr);
        } else {
          // head dimensions rank*64 .. +63 of V_j, all 128 keys
          tma_load_2d_pair(s0, m, 2 * F + h * 128 + rank * 64, jb * BM, bar_addr);
        }
      }
      sc->issued_parity[rp.slot] = static_cast<int>(rp.phase);
      rp.next<NS>();
    }
  }
  return true;
}

// CG = 2 (pair leader): S = Q K^T and O_j = P V are 256-row cta_group::2 MMAs.
// The unit takes both accumulator buffers like two GEMM tiles: S_j alternates
// between the halves of the first, O_j uses the second, so S_{j+1} is computed
// while the epilogue still works on S_j (the ring delivers Q|K of blocks 0 and
// 1, then V_j followed by Q|K of block j+2).
template <int NS, int STAGE_BYTES, int CG>
__device__ bool mma_attn_unit(const KParams& p, SmemCtl<NS>* sc, uint8_t* ring, uint8_t* pbuf, RingPos& rp,
                              uint32_t unit, uint32_t& p_phase, uint32_t& acc, uint32_t& acc_phase) {
  int j0, j1;
  attn_keys<CG>(p.st[unit_stage(unit)], unit, j0, j1);
  const int nkb = j1 - j0;  // key blocks of the unit (even for CG = 2)
  const uint32_t idesc_s = make_idesc_f16(p.bf16, 0, BM * CG, 128);  // Q K^T: both operands K-major
  const uint32_t idesc_o = make_idesc_f16(p.bf16, 1, BM * CG, 128);  // P V: V is MN-major
  const uint32_t pb = smem_u32(pbuf);
  // one full barrier per S buffer: two S in flight must never complete two
  // phases of one barrier before the epilogue has seen the first
  auto mma_s = [&](uint32_t s_tm, uint64_t* s_bar) -> bool {
    for (int part = 0; part < 2; ++part) {
      if (!wait_bar(&sc->full[rp.slot], rp.phase, sc, p, 3)) return false;
      tc_fence_after();
      const uint32_t sa = smem_u32(ring + rp.slot * STAGE_BYTES);
      const uint64_t ad = smem_desc_sw128(sa, 16, 1024), bd = smem_desc_sw128(sa + TILE_A_BYTES, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < BK / UMMA_K; ++kk)
        tc_mma_f16<CG>(s_tm, ad + static_cast<uint64_t>(kk * 2), bd + static_cast<uint64_t>(kk * 2), idesc_s,
                       (part | kk) != 0 ? 1u : 0u);
      tc_commit<CG>(&sc->empty[rp.slot]);
      rp.next<NS>();
    }
    tc_commit<CG>(s_bar);
    return true;
  };
  auto mma_pv = [&](uint32_t o_tm, bool accumulate) -> bool {
    // P_j is in shared memory (of both CTAs) and the previous O_j has been read
    // back; a pair's peer publishes its P with cluster-scope release arrivals
    if (!wait_bar<NS, CG == 2>(&sc->p_full, p_phase, sc, p, 12)) return false;
    p_phase ^= 1u;
    tc_fence_after();
    if (!wait_bar(&sc->full[rp.slot], rp.phase, sc, p, 3)) return false;
    tc_fence_after();
    const uint32_t sv = smem_u32(ring + rp.slot * STAGE_BYTES);
    const uint64_t vd = smem_desc_sw128(sv, TILE_A_BYTES, 1024);  // V: 64-dim atoms 16 KB apart, 8-key groups 1 KB apart
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      // P: chunk of 64 keys per 16 KB, +32 bytes per 16 keys; V: +16 key rows (2 KB)
      const uint64_t a = smem_desc_sw128(pb + (kk >> 2) * (BM * 128), 16, 1024) + static_cast<uint64_t>((kk & 3) * 2);
      tc_mma_f16<CG>(o_tm, a, vd + static_cast<uint64_t>(kk * 128), idesc_o, (accumulate || kk != 0) ? 1u : 0u);
    }
    tc_commit<CG>(&sc->empty[rp.slot]);
    rp.next<NS>();
    tc_commit<CG>(&sc->o_full);
    return true;
  };
  if constexpr (CG == 1) {
    const uint32_t s_tm = sc->tmem_base + ATT_S_COL, o_tm = sc->tmem_base + ATT_O_COL;
    for (int j = 0; j < nkb; ++j)
      if (!mma_s(s_tm, &sc->s_full) || !mma_pv(o_tm, j > 0)) return false;
  } else {
    uint32_t buf[2];
    for (int b = 0; b < 2; ++b) {
      if (!wait_bar(&sc->tempty[acc], acc_phase ^ 1u, sc, p, 2)) return false;
      buf[b] = acc;
      acc ^= 1u;
      if (acc == 0u) acc_phase ^= 1u;
    }
    tc_fence_after();
    const uint32_t stride = static_cast<uint32_t>(p.acc_stride);
    const uint32_t s_base = sc->tmem_base + buf[0] * stride, o_tm = sc->tmem_base + buf[1] * stride;
    if (!mma_s(s_base, &sc->s_full)) return false;
    if (nkb > 1 && !mma_s(s_base + 128, &sc->s_full_b)) return false;
    for (int j = 0; j < nkb; ++j) {
      if (!mma_pv(o_tm, j > 0)) return false;
      // S_j's half is free once P_j is published
      if (j + 2 < nkb && !mma_s(s_base + static_cast<uint32_t>(j & 1) * 128, (j & 1) ? &sc->s_full_b : &sc->s_full))
        return false;
    }
    // hand both buffers back through the GEMM protocol
    tc_commit<CG>(&sc->tfull[buf[0]]);
    tc_commit<CG>(&sc->tfull[buf[1]]);
  }
  return true;
}

// Epilogue warps: online softmax for one query row per thread.  CG = 2: this
// CTA's query block is the unit's block rank; its rows see every key block of
// the unit (the first query block's last one is entirely in its future).
// NE = 8: the two warps of a TMEM lane quadrant share each row, one taking keys
// 0-63 and output dimensions 0-63, the other the rest; they exchange their row
// maxima (and at the end their row sums) through shared memory.
// A piece of a split row ends with its state (m, l and the output scaled by
// 2^-m) in the workspace; the last piece of this query block and head to
// arrive merges all of them in piece order and stores O.
template <int NS, int CG, int NE>
__device__ bool epi_attn_unit(const KParams& p, SmemCtl<NS>* sc, uint8_t* staging, uint32_t unit, uint32_t& s_phase,
                              uint32_t& o_phase, int& last_buf, uint32_t tidx, uint32_t& tacc, uint32_t& tacc_phase,
                              uint32_t rank, uint32_t epoch1) {
  const StageP& S = p.st[unit_stage(unit)];
  const int i = unit_m(unit), h = unit_n(unit);
  const int qb = i * CG + static_cast<int>(rank);  // this CTA's query block
  int j0, j1;
  const int np = attn_keys<CG>(S, unit, j0, j1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;
  const int r = q * 32 + lane;  // query row within the block
  constexpr int NH = NE / 4;    // warps per row
  constexpr int CPW = 4 / NH;   // 32-column chunks of S (keys) and of O (dimensions) per warp
  const int half = (warp - EPI_WARP0) >> 2;
  const int cb = half * CPW;    // this warp's first chunk
  // NE = 8: the other warp of the row's value of x; both have read before
  // either writes the exchange slots again
  auto other = [&](float x) -> float {
    sc->xchg[half][r] = x;
    named_bar_sync(2 + q, 64);
    const float y = sc->xchg[half ^ 1][r];
    named_bar_sync(2 + q, 64);
    return y;
  };
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  // CG = 1: S and O at fixed columns.  CG = 2: S_j in half (j & 1) of the
  // unit's first accumulator buffer, O in its second (the MMA's layout)
  const uint32_t stride = static_cast<uint32_t>(p.acc_stride);
  const uint32_t s_base = sc->tmem_base + lane_base + (CG == 1 ? ATT_S_COL : tacc * stride);
  const uint32_t o_tm = CG == 1 ? sc->tmem_base + lane_base + ATT_O_COL : sc->tmem_base + lane_base + (tacc ^ 1u) * stride;
  const float sl2 = S.softmax_scale_log2;
  float m_ref = -INFINITY, l_run = 0.0f;  // l_run: this warp's keys
  // the staging buffers double as the P operand: earlier stores must be done reading them
  if (lane == 0) tma_store_wait_read<0>();
  __syncwarp();
  last_buf = -1;
  for (int j = j0; j < j1; ++j) {
    // s_phase: bit 0 tracks s_full, bit 1 s_full_b (odd key blocks of pair
    // units; j0 is even there)
    const uint32_t sb = CG == 2 ? static_cast<uint32_t>(j & 1) : 0u;
    if (!wait_bar(sb ? &sc->s_full_b : &sc->s_full, (s_phase >> sb) & 1u, sc, p, 13)) return false;
    s_phase ^= 1u << sb;
    tc_fence_after();
    if (j == j0 && threadIdx.x == EPI_WARP0 * 32) trace_put(p, tidx, rank, CG, 6, globaltimer());
    const uint32_t s_tm = CG == 1 ? s_base : s_base + static_cast<uint32_t>(j & 1) * 128;
    // this warp's part of the row of S_j, read once
    uint32_t v[CPW][32];
#pragma unroll
    for (int c = 0; c < CPW; ++c) tmem_ld32(s_tm + (cb + c) * 32, v[c]);
    tc_wait_ld();
#pragma unroll
    for (int c = 0; c < CPW; ++c) tc_wait_ld_regs(v[c]);
    // scaled logits, -inf where masked: key column k of block j is visible to
    // row r iff j*128 + k <= qb*128 + r
    const bool diag = j >= qb;
    const int lim = (qb - j) * 128 + r;
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < CPW; ++c)
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const float x = (diag && (cb + c) * 32 + t > lim) ? -INFINITY : __uint_as_float(v[c][t]) * sl2;
        v[c][t] = __float_as_uint(x);
        mx[t & 3] = fmaxf(mx[t & 3], x);
      }
    float m_blk = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    if constexpr (NH > 1) m_blk = fmaxf(m_blk, other(m_blk));
    // every row sees a key of the unit's first block (j0 <= qb), so m_ref is
    // finite from then on; both warps of a row take the same decisions
    const bool raise = m_blk > m_ref + ATT_RESCALE_LOG2;
    const float m_new = raise ? m_blk : m_ref;
    if (j > j0) {
      // P V of block j-1 has read P_{j-1} and added into O
      if (!wait_bar(&sc->o_full, o_phase, sc, p, 14)) return false;
      o_phase ^= 1u;
      tc_fence_after();
      if (__any_sync(0xFFFFFFFFu, raise)) {
        // O and l against the raised maximum (tcgen05.ld/st are warp-wide)
        const float f = raise ? ex2_approx(m_ref - m_new) : 1.0f;
        l_run *= f;
#pragma unroll 1
        for (int c = 0; c < CPW; ++c) {
          uint32_t o[32];
          tmem_ld32(o_tm + (cb + c) * 32, o);
          tc_wait_ld();
          tc_wait_ld_regs(o);
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * f);
          tmem_st32(o_tm + (cb + c) * 32, o);
        }
        tc_wait_st();
      }
    }
    m_ref = m_new;
    // P = exp2(s - m_ref) (0 where masked), its row sum, P_j written as the A operand of P V
    float ls[2] = {0.0f, 0.0f};
#pragma unroll
    for (int c = 0; c < CPW; ++c) {
      uint32_t w[16];
#pragma unroll
      for (int t = 0; t < 32; t += 2) {
        const float p0 = ex2_approx(__uint_as_float(v[c][t]) - m_ref);
        const float p1 = ex2_approx(__uint_as_float(v[c][t + 1]) - m_ref);
        ls[0] += p0;
        ls[1] += p1;
        w[t >> 1] = pack2(p0, p1, p.bf16);
      }
      // keys k*32 .. k*32+31 live in 64-key chunk k/2, 16-byte pieces (k%2)*4 .. +3 of row r
      const int k = cb + c;
      uint8_t* rowp = staging + (k >> 1) * (BM * 128) + r * 128;
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        const int piece = (k & 1) * 4 + pc;
        const uint32_t addr = smem_u32(rowp + ((piece ^ (r & 7)) << 4));
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[pc * 4 + 0]),
                     "r"(w[pc * 4 + 1]), "r"(w[pc * 4 + 2]), "r"(w[pc * 4 + 3])
                     : "memory");
      }
    }
    l_run += ls[0] + ls[1];
    fence_proxy_async_shared();
    tc_fence_before();
    if (CG == 1 || rank == 0) {
      // the pair leader's own warps (or a single SM's): one CTA-scope arrival each
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc->p_full);
    } else {
      // the pair's second CTA: every epilogue warp's P is written, then one
      // cluster-scope arrival on the leader's barrier (the leader issues P V)
      named_bar_sync(1, NE * 32);
      if (threadIdx.x == EPI_WARP0 * 32) mbar_arrive_cluster(mapa_shared(&sc->p_full, 0));
    }
  }
  // the last P V, then this warp's O dimensions (against m_ref) into registers
  if (!wait_bar(&sc->o_full, o_phase, sc, p, 14)) return false;
  o_phase ^= 1u;
  tc_fence_after();
  constexpr int DW = CPW * 32;  // output dimensions of this warp: [cb*32, cb*32 + DW)
  float acc[DW];
  {
    uint32_t o[CPW][32];
#pragma unroll
    for (int c = 0; c < CPW; ++c) tmem_ld32(o_tm + (cb + c) * 32, o[c]);
    tc_wait_ld();
#pragma unroll
    for (int c = 0; c < CPW; ++c) {
      tc_wait_ld_regs(o[c]);
#pragma unroll
      for (int t = 0; t < 32; ++t) acc[c * 32 + t] = __uint_as_float(o[c][t]);
    }
  }
  const float m_run = m_ref;
  if constexpr (NH > 1) l_run += other(l_run);  // the row's sum over all 128 keys of every block
  tc_fence_before();
  if constexpr (CG == 2) {
    // every TMEM read of the unit is done: both accumulator buffers go back to
    // the MMA (both CTAs' warps), in order
    for (int b = 0; b < 2; ++b) {
      if (!wait_bar(&sc->tfull[tacc], tacc_phase, sc, p, 4)) return false;
      tc_fence_after();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(&sc->tempty[tacc], 0));
      tacc ^= 1u;
      if (tacc == 0u) tacc_phase ^= 1u;
    }
  }
  if (np > 1) {
    // [piece][ATT_PART_COLS / 4][128 rows] float4: a warp moves 512 contiguous bytes per access
    const size_t piece_floats = static_cast<size_t>(ATT_PART_COLS) * BM;
    float* ws = S.partial + (static_cast<size_t>(qb) * S.n_tiles + h) * S.kv_max * piece_floats;
    float4* mine = reinterpret_cast<float4*>(ws + unit_ks(unit) * piece_floats) + r;
#pragma unroll
    for (int t = 0; t < DW / 4; ++t)
      mine[(cb * 8 + t) * BM] = make_float4(acc[4 * t], acc[4 * t + 1], acc[4 * t + 2], acc[4 * t + 3]);
    if (half == 0) mine[32 * BM] = make_float4(m_run, l_run, 0.0f, 0.0f);
    // as for K-splits: the CTA barrier orders every thread's stores before the
    // one acq_rel arrival; the last piece reads the others' after the next one
    named_bar_sync(1, NE * 32);
    if (threadIdx.x == EPI_WARP0 * 32) {
      const uint32_t old = atom_add_acq_rel_gpu(S.split_ctr + static_cast<size_t>(qb) * S.n_tiles + h, 1u);
      sc->split_last = (old + 1u == epoch1 * static_cast<uint32_t>(np)) ? 1 : 0;
    }
    named_bar_sync(1, NE * 32);
    if (!sc->split_last) {
      if (threadIdx.x == EPI_WARP0 * 32) trace_put(p, tidx, rank, CG, 7, globaltimer());
      return true;
    }
    // O = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k, M = max_k m_k,
    // summed in piece order
    float mx = -INFINITY;
    for (int k = 0; k < np; ++k)
      mx = fmaxf(mx, __ldcg(reinterpret_cast<const float4*>(ws + k * piece_floats) + 32 * BM + r).x);
#pragma unroll
    for (int t = 0; t < DW; ++t) acc[t] = 0.0f;
    float l_sum = 0.0f;
    for (int k = 0; k < np; ++k) {
      const float4* src = reinterpret_cast<const float4*>(ws + k * piece_floats) + r;
      const float4 ml = __ldcg(src + 32 * BM);
      const float w = ex2_approx(ml.x - mx);
      l_sum = fmaf(ml.y, w, l_sum);
#pragma unroll
      for (int c = 0; c < DW / 32; ++c) {
        float4 x[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) x[t] = __ldcg(src + (cb * 8 + c * 8 + t) * BM);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          float* a = &acc[(c * 8 + t) * 4];
          a[0] = fmaf(x[t].x, w, a[0]);
          a[1] = fmaf(x[t].y, w, a[1]);
          a[2] = fmaf(x[t].z, w, a[2]);
          a[3] = fmaf(x[t].w, w, a[3]);
        }
      }
    }
    l_run = l_sum;
  }
  const float inv = 1.0f / l_run;
  // this warp's O dimensions of its rows -> staging (the last P V has completed:
  // P's buffers are free) -> TMA store, 64 dimensions per staging chunk
#pragma unroll
  for (int cc = 0; cc < DW / 64; ++cc) {
    const int c = cb / 2 + cc;
    uint32_t w[32];
#pragma unroll
    for (int t = 0; t < 64; t += 2) w[t >> 1] = pack2(acc[cc * 64 + t] * inv, acc[cc * 64 + t + 1] * inv, p.bf16);
    stage_row(staging, c, r, w);
    fence_proxy_async_shared();
    __syncwarp();
    const int grow = qb * BM + q * 32;
    if (grow < S.m_extent) {
      if (lane == 0) {
        tma_store_2d(&p.maps[S.map_out], staging + c * (BM * 128) + q * 32 * 128, h * 128 + c * 64, grow);
        tma_store_commit();
      }
      last_buf = c;
    }
  }
  if (S.rel_tile != nullptr) {
    release_tile<NE>(p, S, qb, h, lane);
    last_buf = -1;
  }
  if (threadIdx.x == EPI_WARP0 * 32) trace_put(p, tidx, rank, CG, 7, globaltimer());
  return true;
}

// Scheduler poll for an attention unit: items are row blocks 0..i whose Q, K
// and V tiles of head h (TILE / STRIDED) or whose whole row (ROW) are complete.
template <int NS>
__device__ void sched_poll_attn(const KParams& p, const StageP& S, SmemCtl<NS>* sc, uint32_t q, int i, int h,
                                uint32_t epoch1, uint32_t unit, int lane) {
  const int nt = S.dep_ntiles;
  int published = 0;
  const uint64_t t0 = globaltimer();
  uint32_t ns = 64;
  while (true) {
    int ready = i + 1;
    for (int base = 0; base <= i; base += 32) {
      const int j = base + lane;
      bool done = true;
      if (j <= i) {
        if (S.wait == WAIT_ROW) {
          done = static_cast<int32_t>(ld_relaxed_gpu(S.dep_row + j) - epoch1 * static_cast<uint32_t>(nt)) >= 0;
        } else {
          // the producer tile holding columns (part*heads + h)*128 .. +127 (Q, K, V of head h)
#pragma unroll
          for (int part = 0; part < 3; ++part)
            done = done && static_cast<int32_t>(ld_relaxed_gpu(S.dep_tile + static_cast<size_t>(j) * nt +
                                                               (part * S.heads + h) * 128 / S.dep_bn) -
                                                epoch1) >= 0;
        }
      }
      const uint32_t bad = __ballot_sync(0xFFFFFFFFu, !done);
      if (bad) {
        ready = base + __ffs(bad) - 1;
        break;
      }
    }
    if (ready > published) {
      fence_acq_rel_gpu();
      __syncwarp();
      if (lane == 0) st_release_cta_shared(&sc->uq_ready[q], static_cast<uint32_t>(ready));
      published = ready;
    }
    if (published >= i + 1) return;
    bool give_up = false;
    if (lane == 0) {
      if (ld_relaxed_gpu(&p.ctrl[CTRL_ABORT]) != 0u) {
        give_up = true;
      } else if (globaltimer() - t0 > p.timeout_ns) {
        record_error(p, ERR_TIMEOUT, unit, static_cast<uint32_t>(published));
        give_up = true;
      }
    }
    give_up = __shfl_sync(0xFFFFFFFFu, give_up ? 1 : 0, 0) != 0;
    if (give_up) {
      if (lane == 0) st_release_cta_shared(&sc->uq_ready[q], READY_ALL);
      return;
    }
    __nanosleep(ns);
    if (ns < 512) ns <<= 1;
  }
}

// ---------------------------------------------------------------- L2 prefetch
// The scheduler warp spends the time between claims bringing the next K-slices
// of the unit the TMA warp is loading into L2, pf_dist slices ahead of it: the
// weight lines (and a producer's A rows), so that the TMA loads hit in L2
// instead of each stage waiting on its slowest DRAM sector.
struct PfState {
  uint32_t unit = UNIT_END;
  int seq = 0;      // sequence number of that unit in this CTA
  int next = 0;     // next K-slice to prefetch
  int kb0 = 0, kb1 = 0;
};

template <int CG, int CL>
__device__ __forceinline__ void prefetch_slice(const StageP& S, uint32_t unit, int kb, uint32_t rank, int lane) {
  const int m = unit_m(unit), n = unit_n(unit);
  const bool gate_up = CG == 2 && S.pf_b2 != nullptr;
  const int bcols = gate_up ? S.bn : S.bn / CG;
  const int col0 = n * S.bn + (gate_up ? 0 : static_cast<int>(rank & (CG - 1)) * bcols);
  if (S.b_major == 0) {
    // weights [N, K]: one 128-byte line per weight row of the slice
    for (int r = lane; r < bcols; r += 32) {
      const int row = col0 + r;
      if (row < S.pf_brows) {
        const long long off = static_cast<long long>(row) * S.pf_ldb + static_cast<long long>(kb) * BK * 2;
        prefetch_l2(S.pf_b + off);
        if (S.pf_b2) prefetch_l2(S.pf_b2 + off);
      }
    }
  } else {
    // weights [K, N]: 64 K rows of bcols*2 bytes
    const int lines = bcols * 2 / 128;
    for (int i = lane; i < BK * lines; i += 32) {
      const int row = kb * BK + i / lines;
      if (row < S.pf_brows) {
        const long long off = static_cast<long long>(row) * S.pf_ldb + static_cast<long long>(col0) * 2 + (i % lines) * 128;
        prefetch_l2(S.pf_b + off);
        if (S.pf_b2) prefetch_l2(S.pf_b2 + off);
      }
    }
  }
  if (S.pf_a) {
    const int row0 = (m * CL + static_cast<int>(rank)) * BM;
    for (int r = lane; r < BM; r += 32)
      if (row0 + r < S.pf_arows)
        prefetch_l2(S.pf_a + static_cast<long long>(row0 + r) * S.pf_lda + static_cast<long long>(kb) * BK * 2);
  }
}

// Bounded wait for `bar`, prefetching for the latest pushed unit meanwhile.
template <int NS, int CG, int CL, bool CLUSTER>
__device__ bool wait_prefetching(uint64_t* bar, uint32_t parity, SmemCtl<NS>* sc, const KParams& p, PfState& pf,
                                 uint32_t rank, int lane, uint32_t where) {
  if (p.pf_dist <= 0 || pf.unit == UNIT_END || pf.next >= pf.kb1) return wait_bar<NS, CLUSTER>(bar, parity, sc, p, where);
  const StageP& S = p.st[unit_stage(pf.unit)];
  const uint64_t t0 = globaltimer();
  while (true) {
    bool ready = false;
    if (lane == 0) ready = CLUSTER ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity);
    if (__shfl_sync(0xFFFFFFFFu, ready ? 1 : 0, 0)) return true;
    // the TMA warp is on an earlier unit: the first pf_dist slices; else pf_dist ahead of it
    const int limit = min(pf.kb1, (sc->tma_seq < pf.seq ? pf.kb0 : sc->tma_kb + 1) + p.pf_dist);
    while (pf.next < limit) prefetch_slice<CG, CL>(S, pf.unit, pf.next++, rank, lane);
    if (pf.next >= pf.kb1) return wait_bar<NS, CLUSTER>(bar, parity, sc, p, where);
    if (sc->abort) return false;
    if (globaltimer() - t0 > p.watchdog_ns) {
      if (lane == 0) record_error(p, ERR_WATCHDOG, 0xFFFFFFFFu, where);
      sc->abort = 1;
      return false;
    }
    __nanosleep(200);
  }
}

// ---------------------------------------------------------------- scheduler role
template <int NS>
__device__ __forceinline__ void push_unit(SmemCtl<NS>* sc, uint32_t q, uint32_t unit, uint32_t idx, int lane,
                                          bool consumer, uint32_t kb, uint32_t part) {
  if (lane == 0) {
    sc->uq[q] = unit;
    sc->uq_idx[q] = idx;
    sc->uq_kb[q] = kb;
    sc->uq_part[q] = part;
    sc->uq_ready[q] = consumer ? 0u : READY_ALL;
    mbar_arrive(&sc->uq_full[q]);
  }
  __syncwarp();
}

// ---------------------------------------------------------------- the kernel
// ATTN: the instantiation also runs attention units (the attention chain);
// the MLP instantiations leave that code out and keep their registers.
// CG: CTAs per tcgen05 MMA (1, or 2 for a 256-row pair); CL: CTAs per unit
// and per cluster (CG, or 4: two pairs sharing the weight boxes by multicast).
template <int NS, int STAGE_BYTES, int CG, bool ATTN, int CL = CG, int AR = BM>
__global__ void __launch_bounds__(Roles<ATTN>::THREADS, 1) cs_chain_kernel(const __grid_constant__ KParams p) {
  constexpr int NE = Roles<ATTN>::EPI;
  static_assert(CL == CG || (CG == 2 && CL == 4 && !ATTN), "unsupported cluster shape");
#ifdef CS_NO_CLUSTER_MULTICAST
  static_assert(CL != 4, "the replica build has no 4-CTA multicast tiles");
#endif
  static_assert(AR == BM || ((AR == 8 || AR == 32) && CG == 1 && !ATTN),
                "8- and 32-row A tiles are built for single-SM MLP tiles");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* staging = ring + NS * STAGE_BYTES;
  SmemCtl<NS>* sc = reinterpret_cast<SmemCtl<NS>*>(staging + STAGING_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CG == 1 ? 0u : cluster_ctarank();
  const bool leader = rank == 0;                 // claims units for the cluster
  const bool pair_leader = (rank & 1u) == 0u;    // issues the pair's MMAs

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      // one expect_tx arrival per CTA of the pair, on the pair leader's barrier
      // (CL = 4: each pair's leader counts its own pair's bytes)
      mbar_init(&sc->full[i], CG);
      // CL = 4: both pairs' MMAs must be done with a stage before it refills
      mbar_init(&sc->empty[i], CL == 4 ? 2 : 1);
      sc->issued_parity[i] = -1;
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sc->tfull[i], 1);
      mbar_init(&sc->tempty[i], NE * CG);  // every epilogue warp of the tile
    }
    for (int i = 0; i < UQ; ++i) {
      mbar_init(&sc->uq_full[i], 1);
      mbar_init(&sc->uq_empty[i], 2 + NE);  // TMA + MMA + the epilogue warps
    }
    mbar_init(&sc->claim_req, 1);
    mbar_init(&sc->mb_full, 1);
    mbar_init(&sc->mb_empty, CL - 1 > 0 ? CL - 1 : 1);  // every peer CTA takes the index
    mbar_init(&sc->s_full, 1);
    mbar_init(&sc->s_full_b, 1);
    mbar_init(&sc->p_full, CG == 1 ? NE : NE + 1);  // the leader's epilogue warps, one arrival from the peer
    mbar_init(&sc->o_full, 1);
    mbar_init(&sc->drain, 1);
    sc->abort = 0;
    sc->tma_seq = 0;
    sc->tma_kb = 0;
    fence_mbar_init();
    for (int i = 0; i < 9; ++i) prefetch_tmap(&p.maps[i]);
  }
  if (warp == 1) {
    tmem_alloc<CG>(&sc->tmem_base, TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers exist before anyone arrives on them
  tc_fence_after();
  // Everything above touched only this CTA's shared and tensor memory.  Under a
  // programmatic dependent launch the grid queued before this one may still be
  // running: global memory (counters, inputs, outputs) waits for its completion.
  // The next forward may then be scheduled; its CTAs take an SM only when one of
  // this grid's CTAs has left it (each CTA needs most of an SM's shared memory).
  grid_dep_wait();
  grid_dep_launch_dependents();

  const uint32_t epoch1 = p.ctrl[CTRL_EPOCH] + 1u;

  if (warp == Roles<ATTN>::SCHED) {
    uint32_t q = 0, qphase = 0, req_phase = 0, mb_phase = 0;
    bool first = true;
    PfState pf;
    int pushed = 0;
    while (true) {
      uint32_t idx = 0xFFFFFFFFu;  // dispatch index (>= n_units: no more work)
      if (leader) {
        // claim units in schedule order, one at a time, just in time
        if (!first) {
          if (!wait_prefetching<NS, CG, CL, false>(&sc->claim_req, req_phase, sc, p, pf, rank, lane, 9)) break;
          req_phase ^= 1u;
        }
        first = false;
        if (lane == 0 && ld_relaxed_gpu(&p.ctrl[CTRL_ABORT]) == 0u) idx = atomicAdd(&p.ctrl[CTRL_DISPATCH], 1u);
        idx = __shfl_sync(0xFFFFFFFFu, idx, 0);
        if constexpr (CG == 2) {
          // hand the dispatch index to the other CTAs of the cluster
          if (!wait_bar<NS, true>(&sc->mb_empty, mb_phase ^ 1u, sc, p, 10)) break;
          if (lane > 0 && lane < CL) {
            st_cluster_u32(mapa_shared(&sc->mb_unit, static_cast<uint32_t>(lane)), idx);
            mbar_arrive_cluster(mapa_shared(&sc->mb_full, static_cast<uint32_t>(lane)));
          }
          __syncwarp();
          mb_phase ^= 1u;
        }
      } else {
        if (!wait_prefetching<NS, CG, CL, true>(&sc->mb_full, mb_phase, sc, p, pf, rank, lane, 11)) break;
        idx = *reinterpret_cast<volatile uint32_t*>(&sc->mb_unit);
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(&sc->mb_empty, 0));
        mb_phase ^= 1u;
      }
      const uint32_t unit = idx < static_cast<uint32_t>(p.n_units) ? p.sched[idx] : UNIT_END;
      if (unit != UNIT_END && lane == 0) {
        trace_put(p, idx, rank, CL, 0, unit | (static_cast<unsigned long long>(idx) << 32));
        trace_put(p, idx, rank, CL, 1, smid() | (blockIdx.x << 16) | (rank << 30));
        trace_put(p, idx, rank, CL, 2, globaltimer());
      }
      if (unit == UNIT_END) {
        if (wait_bar(&sc->uq_empty[q], qphase ^ 1u, sc, p, 5))
          push_unit(sc, q, UNIT_END, idx, lane, false, 0u, PART_TILE | PART_LAST);
        break;
      }
      const StageP& S = p.st[unit_stage(unit)];
      const bool consumer = p.waits && S.wait != WAIT_NONE;
      // The claimed unit's pieces: one for a tile unit; for Stream-K unit u,
      // one per tile that its K-slices [u*q, (u+1)*q) of the SK tiles'
      // concatenated K ranges touch (contributor u - first of that tile).
      const bool sk = S.kind == STAGE_GEMM && unit_ks(unit) == SK_KS;
      const long long K = S.k_iters;
      const long long sk_a = sk ? static_cast<long long>(unit_n(unit)) * S.sk_q : 0;
      const long long sk_b = sk ? min(static_cast<long long>(S.sk_tiles) * K, sk_a + S.sk_q) : 0;
      int j = sk ? static_cast<int>(sk_a / K) : 0;
      const int j_end = sk ? static_cast<int>((sk_b - 1) / K) + 1 : 1;
      bool ok = true;
      for (; j < j_end; ++j) {
        uint32_t pu = unit, kb = 0u, part = PART_TILE | PART_LAST | (1u << 8);
        if (sk) {
          pu = S.sk_tile[j];
          const long long t0 = j * K;
          const int kb0 = static_cast<int>(max(sk_a, t0) - t0), kb1 = static_cast<int>(min(sk_b, t0 + K) - t0);
          const int first = static_cast<int>(t0 / S.sk_q), last = static_cast<int>((t0 + K - 1) / S.sk_q);
          kb = static_cast<uint32_t>(kb0) | (static_cast<uint32_t>(kb1) << 16);
          part = static_cast<uint32_t>(unit_n(unit) - first) | (static_cast<uint32_t>(last - first + 1) << 8) |
                 (j + 1 == j_end ? PART_LAST : 0u) | (static_cast<uint32_t>(j) << 16);
        } else if (S.kind == STAGE_GEMM) {
          const int kb0 = unit_ks(unit) * S.kps, kb1 = min(S.k_iters, kb0 + S.kps);
          kb = static_cast<uint32_t>(kb0) | (static_cast<uint32_t>(kb1) << 16);
          part = static_cast<uint32_t>(unit_ks(unit)) | (static_cast<uint32_t>(S.splits) << 8) | PART_LAST | PART_TILE;
        }
        if (!wait_bar(&sc->uq_empty[q], qphase ^ 1u, sc, p, 5)) {
          ok = false;
          break;
        }
        push_unit(sc, q, pu, idx, lane, consumer, kb, part);
        ++pushed;
        if (S.kind == STAGE_GEMM && S.pf_b != nullptr) {
          pf.unit = pu;
          pf.seq = pushed;
          pf.kb0 = piece_kb0(kb);
          pf.kb1 = piece_kb1(kb);
          pf.next = pf.kb0;
        } else {
          pf.unit = UNIT_END;
        }
        if (consumer && S.kind == STAGE_GEMM)
          sched_poll_gemm<NS>(p, S, sc, q, unit_m(pu) * CL + static_cast<int>(rank), epoch1, pu, piece_kb0(kb),
                              piece_kb1(kb), lane);
        else if constexpr (ATTN)
          if (consumer && S.kind == STAGE_ATTN)
            sched_poll_attn<NS>(p, S, sc, q, (unit_m(pu) + 1) * CG - 1, unit_n(pu), epoch1, pu, lane);
        if (lane == 0) trace_put(p, idx, rank, CL, 3, globaltimer());
        if (++q == UQ) {
          q = 0;
          qphase ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else if (warp == 0) {
    if (lane == 0) {
      RingPos rp;
      uint32_t q = 0, qphase = 0;
      bool ok = true;
      while (ok) {
        if (!wait_bar(&sc->uq_full[q], qphase, sc, p, 6)) break;
        const uint32_t unit = sc->uq[q];
        if (unit != UNIT_END && p.st[unit_stage(unit)].kind == STAGE_GEMM)
          ok = tma_gemm_unit<NS, STAGE_BYTES, CG, CL, AR>(p, sc, ring, rp, unit, q, rank);
        else if constexpr (ATTN)
          if (unit != UNIT_END) ok = tma_attn_unit<NS, STAGE_BYTES, CG>(p, sc, ring, rp, unit, q, rank);
        mbar_arrive(&sc->uq_empty[q]);
        if (++q == UQ) {
          q = 0;
          qphase ^= 1u;
        }
        if (unit == UNIT_END) break;
      }
      // Let every load this thread issued land before the CTA can exit.  In
      // pair mode (and CL = 4) the loads complete on the pair leader's barrier,
      // which its MMA waits for; after an abort, give in-flight copies a bounded
      // grace time.
      if constexpr (CG == 1) {
        for (int i = 0; i < NS; ++i)
          if (sc->issued_parity[i] >= 0) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(&sc->full[i], static_cast<uint32_t>(sc->issued_parity[i])) &&
                   globaltimer() - t0 < p.watchdog_ns) {
            }
          }
      } else if (!ok) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 200000u) __nanosleep(1000);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      RingPos rp;
      uint32_t q = 0, qphase = 0, acc = 0, acc_phase = 0, p_phase = 0;
      bool ok = true;
      bool issued = false;
      while (ok) {
        if (!wait_bar(&sc->uq_full[q], qphase, sc, p, 6)) break;
        const uint32_t unit = sc->uq[q];
        const uint32_t kb = sc->uq_kb[q];
        mbar_arrive(&sc->uq_empty[q]);
        if (++q == UQ) {
          q = 0;
          qphase ^= 1u;
        }
        if (unit == UNIT_END) break;
        if (p.st[unit_stage(unit)].kind == STAGE_GEMM) {
          if (pair_leader) {
            ok = mma_gemm_unit<NS, STAGE_BYTES, CG, CL, AR>(p, sc, ring, rp, unit, piece_kb0(kb), piece_kb1(kb), acc,
                                                            acc_phase, rank);
            issued = true;
          }
        } else if constexpr (ATTN) {
          if (pair_leader) {
            ok = mma_attn_unit<NS, STAGE_BYTES, CG>(p, sc, ring, staging, rp, unit, p_phase, acc, acc_phase);
            issued = true;
          }
        }
      }
      // every MMA this thread issued completes before TMEM is freed
      if (issued) {
        if constexpr (CG == 1)
          tc_commit<1>(&sc->drain);
        else
          tc_commit_local_pair(&sc->drain);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&sc->drain, 0) && globaltimer() - t0 < p.watchdog_ns) {
        }
      }
    }
  } else {
    uint32_t q = 0, qphase = 0, acc = 0, acc_phase = 0, s_phase = 0, o_phase = 0;
    int last_buf = -1;  // staging buffer read by this warp's newest committed store
    bool ok = true;
    while (ok) {
      if (!wait_bar(&sc->uq_full[q], qphase, sc, p, 7)) break;
      const uint32_t unit = sc->uq[q];
      const uint32_t tidx = sc->uq_idx[q];
      const uint32_t part = sc->uq_part[q];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc->uq_empty[q]);
      if (++q == UQ) {
        q = 0;
        qphase ^= 1u;
      }
      if (unit == UNIT_END) break;
      if (p.st[unit_stage(unit)].kind == STAGE_GEMM)
        ok = epi_gemm_unit<NS, CG, CL, NE, !ATTN>(p, sc, staging, unit, part, acc, acc_phase, last_buf, rank, tidx,
                                                  epoch1);
      else if constexpr (ATTN)
        ok = epi_attn_unit<NS, CG, NE>(p, sc, staging, unit, s_phase, o_phase, last_buf, tidx, acc, acc_phase, rank,
                                       epoch1);
    }
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // no CTA of a pair leaves while its peer may still signal its barriers or
  // read its shared memory through the pair MMA
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<CG>(sc->tmem_base, TMEM_COLS);

  // Last CTA out re-arms the dispatch counter for the next launch on this
  // stream and, when this launch completes a forward, advances the epoch.
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(&p.ctrl[CTRL_EXIT], 1u);
    if (prev == gridDim.x - 1) {
      p.ctrl[CTRL_DISPATCH] = 0u;
      p.ctrl[CTRL_EXIT] = 0u;
      if (p.bump_epoch && ld_relaxed_gpu(&p.ctrl[CTRL_ERROR]) == 0u) p.ctrl[CTRL_EPOCH] = p.ctrl[CTRL_EPOCH] + 1u;
      __threadfence();
    }
  }
}

}  // namespace cs
