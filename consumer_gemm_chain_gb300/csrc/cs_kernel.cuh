// Persistent tile-synchronised GEMM-chain kernel for sm_103a.
//
// One CTA per SM pulls work units from a dependency-ordered schedule through a
// global atomic counter (a megakernel-style task queue: a dependent task starts
// once the slice it reads is done, not when the whole producer op is done).
// Roles inside a CTA (192 threads):
//   warp 0      : dispatcher + TMA producer (lane 0).  For consumer units it
//                 acquire-spins on the producer tile semaphores of each K-slice
//                 before issuing the TMA loads of the intermediate.
//   warp 1      : TMEM allocator (whole warp) and tcgen05.mma issuer (lane 0).
//   warps 2..5  : epilogue: tcgen05.ld of the fp32 accumulator, bias + GeLU /
//                 SiLU*up / none, downcast, swizzled smem staging, TMA store,
//                 then (producer stages) release-increment of the tile
//                 semaphore and of the row counter.
// Every wait is bounded: semaphore spins by the plan's timeout (error word +
// global abort flag), mbarrier waits by a watchdog (error word + CTA abort).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cs_ptx.cuh"

namespace cs {

constexpr int BM = 128;           // tile rows (UMMA M)
constexpr int BK = 64;            // K-slice per pipeline stage (128 bytes of fp16/bf16)
constexpr int UMMA_K = 16;        // K per tcgen05.mma (kind::f16)
constexpr int TILE_A_BYTES = BM * BK * 2;  // 16 KB
constexpr int STAGING_BYTES = 2 * BM * 128;  // two 64-column chunks of a 128x128 tile
constexpr int UQ = 4;             // unit-queue depth (dispatcher -> MMA/epilogue)
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int EPI_THREADS = 128;
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
  int m_tiles, n_tiles;
  int k_iters;     // BK-slices of the reduction
  int n_extent;    // valid output columns (bias guard, store guard)
  int m_extent;    // valid output rows (store guard)
  int bn;          // output columns per tile (128 or 256)
  int mma_n;       // UMMA N (bn, or 256 for gate|up with bn = 128)
  int b_major;     // 0: weights K-major ([N,K]); 1: MN-major ([K,N])
  int map_a, map_b, map_b2, map_out;
  int b_bytes;     // bytes of the B operand per pipeline stage
  const __nv_bfloat16* bias_bf16;  // exactly one of these two is used (per dtype)
  const __half* bias_f16;
  // consumer side
  int wait;        // WAIT_*
  const uint32_t* dep_tile;  // producer tile semaphores [m_tiles][dep_ntiles]
  const uint32_t* dep_row;   // producer row counters [m_tiles]
  int dep_ntiles;
  int dep_bn;      // intermediate columns per producer tile
  int stride;      // WAIT_STRIDED stride (producer column tiles)
  // producer side
  uint32_t* rel_tile;  // this stage's tile semaphores (null: no release)
  uint32_t* rel_row;
  const uint32_t* delay_ns;  // per unit m*n_tiles+n, or null
  int skip_unit;   // unit that skips its release (-1: none)
  // attention (STAGE_ATTN)
  int heads;
  float softmax_scale_log2;  // log2(e) / sqrt(head_dim)
};

struct KParams {
  CUtensorMap maps[8];
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
};

template <int NS>
struct SmemCtl {
  uint64_t full[NS], empty[NS];
  uint64_t tfull[2], tempty[2];
  uint64_t uq_full[UQ], uq_empty[UQ];
  uint64_t s_full, s_empty, p_full, o_full, o_empty;
  uint64_t drain;
  uint32_t uq[UQ];
  uint32_t tmem_base;
  volatile int abort;
  int issued_parity[NS];  // TMA thread: parity of the last load issued into each slot (-1: none)
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
template <int NS>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, SmemCtl<NS>* sc, const KParams& p,
                                         uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  uint32_t it = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (sc->abort) return false;
    if ((++it & 63u) == 0u && globaltimer() - t0 > p.watchdog_ns) {
      record_error(p, ERR_WATCHDOG, 0xFFFFFFFFu, where);
      sc->abort = 1;
      return false;
    }
  }
}

// Bounded acquire-spin until *ptr >= target (wrap-safe).  False on timeout or
// global abort; the caller then proceeds without the data (the call's result is
// void and cs_chain_status reports the error).
__device__ __forceinline__ bool spin_geq(const uint32_t* ptr, uint32_t target, const KParams& p, uint32_t unit,
                                         uint32_t where) {
  if (static_cast<int32_t>(ld_acquire_gpu(ptr) - target) >= 0) return true;
  const uint64_t t0 = globaltimer();
  uint32_t ns = 32;
  while (true) {
    __nanosleep(ns);
    if (ns < 256) ns <<= 1;
    if (static_cast<int32_t>(ld_acquire_gpu(ptr) - target) >= 0) return true;
    if (ld_relaxed_gpu(&p.ctrl[CTRL_ABORT]) != 0u) return false;
    if (globaltimer() - t0 > p.timeout_ns) {
      record_error(p, ERR_TIMEOUT, unit, where);
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t unit_stage(uint32_t u) { return u >> 28; }
__device__ __forceinline__ int unit_m(uint32_t u) { return static_cast<int>((u >> 14) & 0x3FFFu); }
__device__ __forceinline__ int unit_n(uint32_t u) { return static_cast<int>(u & 0x3FFFu); }

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

// Wait until producer tile column `t` of row block `m` may be read, under the
// stage's policy.  `epoch1` = number of this forward (completed forwards + 1).
__device__ __forceinline__ void wait_gemm_dep(const KParams& p, const StageP& S, int m, int t, uint32_t epoch1,
                                              uint32_t unit, bool first) {
  bool waited = false;
  if (S.wait == WAIT_TILE) {
    spin_geq(S.dep_tile + static_cast<size_t>(m) * S.dep_ntiles + t, epoch1, p, unit, static_cast<uint32_t>(t));
    waited = true;
  } else if (S.wait == WAIT_ROW) {
    if (first) {
      spin_geq(S.dep_row + m, epoch1 * static_cast<uint32_t>(S.dep_ntiles), p, unit, 0x10000u);
      waited = true;
    }
  } else if (S.wait == WAIT_STRIDED) {
    for (int tt = t % S.stride; tt < S.dep_ntiles; tt += S.stride)
      spin_geq(S.dep_tile + static_cast<size_t>(m) * S.dep_ntiles + tt, epoch1, p, unit, static_cast<uint32_t>(tt));
    waited = true;
  }
  // The intermediate was written through the async proxy (TMA store) on other
  // SMs and will be read through the async proxy (TMA load) here.
  if (waited) fence_proxy_async_global();
}

// ---------------------------------------------------------------- TMA role
template <int NS, int STAGE_BYTES>
__device__ bool tma_gemm_unit(const KParams& p, SmemCtl<NS>* sc, uint8_t* ring, RingPos& rp, uint32_t unit,
                              uint32_t epoch1) {
  const StageP& S = p.st[unit_stage(unit)];
  const int m = unit_m(unit), n = unit_n(unit);
  const uint32_t bytes = TILE_A_BYTES + S.b_bytes;
  const bool do_wait = p.waits && S.wait != WAIT_NONE;
  int last_t = -1;
  for (int kb = 0; kb < S.k_iters; ++kb) {
    if (do_wait) {
      const int t = (kb * BK) / S.dep_bn;
      if (t != last_t) {
        wait_gemm_dep(p, S, m, t, epoch1, unit, last_t < 0);
        last_t = t;
      }
    }
    if (!wait_bar(&sc->empty[rp.slot], rp.phase ^ 1u, sc, p, 1)) return false;
    uint8_t* sa = ring + rp.slot * STAGE_BYTES;
    uint8_t* sb = sa + TILE_A_BYTES;
    uint64_t* bar = &sc->full[rp.slot];
    mbar_arrive_expect_tx(bar, bytes);
    tma_load_2d(sa, &p.maps[S.map_a], kb * BK, m * BM, bar);
    // B operand(s): bn rows of N per operand; a second operand (the up
    // projection of gate|up) follows the first, so one N = 2*bn MMA covers both.
    const int nops = S.map_b2 >= 0 ? 2 : 1;
    for (int op = 0; op < nops; ++op) {
      const CUtensorMap* bm = &p.maps[op == 0 ? S.map_b : S.map_b2];
      uint8_t* dst = sb + op * S.bn * (BK * 2);
      if (S.b_major == 0) {
        // weights [N, K]: boxes of 64 K x 128 N rows (16 KB), stacked along N
        for (int h = 0; h < S.bn / 128; ++h) tma_load_2d(dst + h * 16384, bm, kb * BK, n * S.bn + h * 128, bar);
      } else {
        // weights [K, N]: boxes of 64 N (contiguous) x 64 K rows (8 KB), one per 64 columns
        for (int h = 0; h < S.bn / 64; ++h) tma_load_2d(dst + h * 8192, bm, n * S.bn + h * 64, kb * BK, bar);
      }
    }
    sc->issued_parity[rp.slot] = static_cast<int>(rp.phase);
    rp.next<NS>();
  }
  return true;
}

// ---------------------------------------------------------------- MMA role
template <int NS, int STAGE_BYTES>
__device__ bool mma_gemm_unit(const KParams& p, SmemCtl<NS>* sc, uint8_t* ring, RingPos& rp, uint32_t unit,
                              uint32_t& acc, uint32_t& acc_phase) {
  const StageP& S = p.st[unit_stage(unit)];
  const uint32_t idesc = make_idesc_f16(p.bf16, S.b_major, BM, S.mma_n);
  if (!wait_bar(&sc->tempty[acc], acc_phase ^ 1u, sc, p, 2)) return false;
  tc_fence_after();
  const uint32_t d = sc->tmem_base + acc * static_cast<uint32_t>(p.acc_stride);
  for (int kb = 0; kb < S.k_iters; ++kb) {
    if (!wait_bar(&sc->full[rp.slot], rp.phase, sc, p, 3)) return false;
    tc_fence_after();
    const uint32_t sa = smem_u32(ring + rp.slot * STAGE_BYTES);
    const uint32_t sb = sa + TILE_A_BYTES;
    const uint64_t adesc = smem_desc_sw128(sa, 16, 1024);
    // K-major B: 8-row groups 1024 B apart.  MN-major B: 64-column atoms 8 KB
    // apart (LBO), 8-row K groups 1024 B apart (SBO).
    const uint64_t bdesc = S.b_major == 0 ? smem_desc_sw128(sb, 16, 1024) : smem_desc_sw128(sb, 8192, 1024);
#pragma unroll
    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
      const uint64_t a = adesc + static_cast<uint64_t>(kk * 2);  // +32 bytes along K
      const uint64_t b = bdesc + static_cast<uint64_t>(S.b_major == 0 ? kk * 2 : kk * 128);  // +32 B / +16 rows
      tc_mma_f16(d, a, b, idesc, (kb | kk) != 0 ? 1u : 0u);
    }
    tc_commit(&sc->empty[rp.slot]);
    rp.next<NS>();
  }
  tc_commit(&sc->tfull[acc]);
  acc ^= 1u;
  if (acc == 0u) acc_phase ^= 1u;
  return true;
}

// ---------------------------------------------------------------- epilogue role
__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float k1 = 0.044715f;
  return 0.5f * x * (1.0f + tanhf(k0 * (x + k1 * x * x * x)));
}
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ uint32_t pack2(float a, float b, int bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float load_bias(const StageP& S, int col, int bf16) {
  if (col >= S.n_extent) return 0.0f;
  return bf16 ? __bfloat162float(S.bias_bf16[col]) : __half2float(S.bias_f16[col]);
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
// publishes the tile (and its row) with gpu-scope release semantics.
template <int NS>
__device__ void release_tile(const KParams& p, const StageP& S, SmemCtl<NS>* sc, int m, int n, int lane) {
  (void)sc;
  if (lane == 0) {
    tma_store_wait_all<0>();
    fence_proxy_async_global();
  }
  named_bar_sync(1, EPI_THREADS);
  if (threadIdx.x == EPI_WARP0 * 32) {
    const int u = m * S.n_tiles + n;
    if (S.delay_ns != nullptr) {
      const uint64_t d = S.delay_ns[u] > 10000000u ? 10000000u : S.delay_ns[u];
      if (d) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < d) __nanosleep(256);
      }
    }
    if (p.release && S.rel_tile != nullptr && u != S.skip_unit) {
      __threadfence();
      red_release_gpu_add(S.rel_tile + u, 1u);
      red_release_gpu_add(S.rel_row + m, 1u);
    }
  }
}

template <int NS>
__device__ bool epi_gemm_unit(const KParams& p, SmemCtl<NS>* sc, uint8_t* staging, uint32_t unit, uint32_t& acc,
                              uint32_t& acc_phase, int& last_buf) {
  const StageP& S = p.st[unit_stage(unit)];
  const int m = unit_m(unit), n = unit_n(unit);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lane quadrant this warp may access
  const int row = q * 32 + lane;
  if (!wait_bar(&sc->tfull[acc], acc_phase, sc, p, 4)) return false;
  tc_fence_after();
  const uint32_t tbase = sc->tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * static_cast<uint32_t>(p.acc_stride);
  const int nchunks = S.bn / 64;
#pragma unroll 1
  for (int c = 0; c < nchunks; ++c) {
    uint32_t v[2][32];
    uint32_t u[2][32];
    tmem_ld32(tbase + c * 64, v[0]);
    tmem_ld32(tbase + c * 64 + 32, v[1]);
    if (S.epi == EPI_SWIGLU) {
      tmem_ld32(tbase + S.bn + c * 64, u[0]);
      tmem_ld32(tbase + S.bn + c * 64 + 32, u[1]);
    }
    tc_wait_ld();
    if (c == nchunks - 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc->tempty[acc]);
    }
    uint32_t w[32];
    const int col0 = n * S.bn + c * 64;
#pragma unroll
    for (int j = 0; j < 64; j += 2) {
      float a = __uint_as_float(v[j >> 5][j & 31]);
      float b = __uint_as_float(v[(j + 1) >> 5][(j + 1) & 31]);
      if (S.epi == EPI_BIAS_GELU) {
        a = gelu_tanh_f(a + load_bias(S, col0 + j, p.bf16));
        b = gelu_tanh_f(b + load_bias(S, col0 + j + 1, p.bf16));
      } else if (S.epi == EPI_SWIGLU) {
        a = silu_f(a) * __uint_as_float(u[j >> 5][j & 31]);
        b = silu_f(b) * __uint_as_float(u[(j + 1) >> 5][(j + 1) & 31]);
      }
      w[j >> 1] = pack2(a, b, p.bf16);
    }
    // Two chunk buffers alternate.  Every earlier store that read this buffer
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
    stage_row(staging, buf, row, w);
    fence_proxy_async_shared();
    __syncwarp();
    // boxes that start past the tensor's end are skipped, not clipped
    if (col0 < S.n_extent && m * BM + q * 32 < S.m_extent) {
      if (lane == 0) {
        tma_store_2d(&p.maps[S.map_out], staging + buf * (BM * 128) + q * 32 * 128, col0, m * BM + q * 32);
        tma_store_commit();
      }
      last_buf = buf;
    }
  }
  acc ^= 1u;
  if (acc == 0u) acc_phase ^= 1u;
  if (S.rel_tile != nullptr) {
    release_tile(p, S, sc, m, n, lane);
    last_buf = -1;
  }
  return true;
}

// ---------------------------------------------------------------- the kernel
template <int NS, int STAGE_BYTES>
__global__ void __launch_bounds__(NUM_THREADS, 1) cs_chain_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* staging = ring + NS * STAGE_BYTES;
  SmemCtl<NS>* sc = reinterpret_cast<SmemCtl<NS>*>(staging + STAGING_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sc->full[i], 1);
      mbar_init(&sc->empty[i], 1);
      sc->issued_parity[i] = -1;
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sc->tfull[i], 1);
      mbar_init(&sc->tempty[i], 4);
    }
    for (int i = 0; i < UQ; ++i) {
      mbar_init(&sc->uq_full[i], 1);
      mbar_init(&sc->uq_empty[i], 5);
    }
    mbar_init(&sc->s_full, 1);
    mbar_init(&sc->s_empty, 4);
    mbar_init(&sc->p_full, 4);
    mbar_init(&sc->o_full, 1);
    mbar_init(&sc->o_empty, 4);
    mbar_init(&sc->drain, 1);
    sc->abort = 0;
    fence_mbar_init();
    for (int i = 0; i < 8; ++i) prefetch_tmap(&p.maps[i]);
  }
  if (warp == 1) {
    tmem_alloc(&sc->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t epoch1 = p.ctrl[CTRL_EPOCH] + 1u;

  if (warp == 0) {
    if (lane == 0) {
      RingPos rp;
      uint32_t q = 0, qphase = 0;
      bool ok = true;
      while (ok) {
        uint32_t unit = UNIT_END;
        if (ld_relaxed_gpu(&p.ctrl[CTRL_ABORT]) == 0u) {
          const uint32_t idx = atomicAdd(&p.ctrl[CTRL_DISPATCH], 1u);
          if (idx < static_cast<uint32_t>(p.n_units)) unit = p.sched[idx];
        }
        if (!wait_bar(&sc->uq_empty[q], qphase ^ 1u, sc, p, 5)) break;
        sc->uq[q] = unit;
        mbar_arrive(&sc->uq_full[q]);
        if (++q == UQ) {
          q = 0;
          qphase ^= 1u;
        }
        if (unit == UNIT_END) break;
        if (p.st[unit_stage(unit)].kind == STAGE_GEMM)
          ok = tma_gemm_unit<NS, STAGE_BYTES>(p, sc, ring, rp, unit, epoch1);
      }
      // let every load this thread issued land before the CTA can exit
      for (int i = 0; i < NS; ++i)
        if (sc->issued_parity[i] >= 0) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(&sc->full[i], static_cast<uint32_t>(sc->issued_parity[i])) &&
                 globaltimer() - t0 < p.watchdog_ns) {
          }
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      RingPos rp;
      uint32_t q = 0, qphase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      while (ok) {
        if (!wait_bar(&sc->uq_full[q], qphase, sc, p, 6)) break;
        const uint32_t unit = sc->uq[q];
        mbar_arrive(&sc->uq_empty[q]);
        if (++q == UQ) {
          q = 0;
          qphase ^= 1u;
        }
        if (unit == UNIT_END) break;
        if (p.st[unit_stage(unit)].kind == STAGE_GEMM)
          ok = mma_gemm_unit<NS, STAGE_BYTES>(p, sc, ring, rp, unit, acc, acc_phase);
      }
      // every MMA this thread issued completes before TMEM is freed
      tc_commit(&sc->drain);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&sc->drain, 0) && globaltimer() - t0 < p.watchdog_ns) {
      }
    }
  } else {
    uint32_t q = 0, qphase = 0, acc = 0, acc_phase = 0;
    int last_buf = -1;  // staging buffer read by this warp's newest committed store
    bool ok = true;
    while (ok) {
      if (!wait_bar(&sc->uq_full[q], qphase, sc, p, 7)) break;
      const uint32_t unit = sc->uq[q];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc->uq_empty[q]);
      if (++q == UQ) {
        q = 0;
        qphase ^= 1u;
      }
      if (unit == UNIT_END) break;
      if (p.st[unit_stage(unit)].kind == STAGE_GEMM)
        ok = epi_gemm_unit<NS>(p, sc, staging, unit, acc, acc_phase, last_buf);
    }
    if (lane == 0) tma_store_wait_all<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(sc->tmem_base, TMEM_COLS);

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
