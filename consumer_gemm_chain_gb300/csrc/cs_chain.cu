// Host side of the C ABI declared in include/cs_chain.h: plan construction,
// dependency-ordered schedule, TMA descriptor encoding, launches and status.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/cs_chain.h"
#include "cs_kernel.cuh"
#include "cs_sched.cuh"
#include "cs_tune.h"

namespace {

thread_local char g_err[512] = "";

cs_status fail(cs_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

#define CS_CUDA(call)                                                                              \
  do {                                                                                             \
    cudaError_t e_ = (call);                                                                       \
    if (e_ != cudaSuccess) return fail(CS_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_));     \
  } while (0)

constexpr int kMaxMaps = 9;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
// The replica build (CS_NO_CLUSTER_MULTICAST), which processes that share a
// node with other GPUs' ranks load, has no 512-row tiles: those are the only
// ones whose weight boxes travel by TMA cluster multicast.
#ifdef CS_NO_CLUSTER_MULTICAST
constexpr bool kClusterMulticast = false;
#else
constexpr bool kClusterMulticast = true;
#endif

// Kernel configurations: ring depth x stage bytes.  A stage holds the A slice
// (128 x 64) and the B slice (128 x 64; or 256 x 64 for 256-wide tiles and for
// gate|up).  Both rings keep 192 KB of operands in flight per SM.
constexpr int NS_A = 6, SB_A = cs::TILE_A_BYTES + 128 * cs::BK * 2;      // 32 KB stages
constexpr int NS_B = 4, SB_B = cs::TILE_A_BYTES + 2 * 128 * cs::BK * 2;  // 48 KB stages
// up to 8 rows: 8-row A tiles (1 KB) leave room for deeper rings of weights
constexpr int NS_S = 11, SB_S = 8 * cs::BK * 2 + 128 * cs::BK * 2;      // 17 KB stages
constexpr int NS_T = 5, SB_T = 8 * cs::BK * 2 + 2 * 128 * cs::BK * 2;   // 33 KB stages
// 9 to 32 rows: 32-row A tiles (4 KB), 9 stages of 128 weight rows (144 KB in
// flight against 96 KB with 128-row A tiles) or 5 of 256
constexpr int NS_U = 9, SB_U = 32 * cs::BK * 2 + 128 * cs::BK * 2;      // 20 KB stages
constexpr int NS_V = 5, SB_V = 32 * cs::BK * 2 + 2 * 128 * cs::BK * 2;  // 36 KB stages

template <int NS, int SB>
constexpr int smem_bytes_for() {
  return NS * SB + cs::STAGING_BYTES + static_cast<int>(sizeof(cs::SmemCtl<NS>)) + 1024;
}
// every configuration fits the 227 KB a CTA may use
static_assert(smem_bytes_for<NS_A, SB_A>() <= 232448 && smem_bytes_for<NS_B, SB_B>() <= 232448 &&
                  smem_bytes_for<NS_S, SB_S>() <= 232448 && smem_bytes_for<NS_T, SB_T>() <= 232448 &&
                  smem_bytes_for<NS_U, SB_U>() <= 232448 && smem_bytes_for<NS_V, SB_V>() <= 232448,
              "shared memory");

struct MapSlot {
  const void* ptr = nullptr;  // caller pointer the map was encoded for (nullptr: plan-owned or unset)
  bool valid = false;
};

}  // namespace

cs_status cs_fail(cs_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

struct cs_chain_s {
  cs_chain_desc d{};  // as run: tuning-table choices applied, policy AUTO resolved
  int tuned_entry = -1;
  int device = 0;
  int num_sms = 0;
  int m_tiles = 0;
  int stages = 0;
  int n_tiles[3] = {0, 0, 0};
  int k_iters[3] = {0, 0, 0};
  int units[3] = {0, 0, 0};
  int lag = 0;
  int group_m = 1;
  int raster = 1;  // order used: 1 column-major, 2 row-major, 3 K-range-major split consumers
  int stride = 1;
  int bn[3] = {128, 128, 128};
  int cfg_b = 0;  // 1: 48 KB-stage kernel (256-wide one-SM tiles or gate|up)
  int cfg_s = 0;  // up to 8 rows: 1 = 11 x 17 KB stages (128-wide B), 2 = 5 x 33 KB (256 rows of B);
                  // 9 to 32 rows: 3 = 9 x 20 KB, 4 = 5 x 36 KB (measured: GPT-3 M=32
                  // 66.3 -> 63.7 us, stress M=32 73.7 -> 70.3; 64-row A tiles with 7 x 24 KB
                  // stages for 33 to 64 rows changed nothing)
  // cs_mlp_forward_host: double-buffered device X / Y, copy streams and events
  void* host_x[2] = {nullptr, nullptr};
  void* host_y[2] = {nullptr, nullptr};
  cudaStream_t s_h2d = nullptr, s_d2h = nullptr;
  cudaEvent_t ev_x[2] = {nullptr, nullptr}, ev_k[2] = {nullptr, nullptr}, ev_y[2] = {nullptr, nullptr};
  unsigned long long host_calls = 0;
  int cg = 1;     // CTAs per tcgen05 MMA (2: 256-row tiles on a 2-SM pair)
  int cl = 1;     // CTAs per unit and cluster (4: two pairs sharing weight boxes)
  int m_units = 0;   // tile rows of the schedule
  int m_blocks = 0;  // 128-row blocks (semaphore rows)
  int sched_units[3] = {0, 0, 0};
  int splits[3] = {1, 1, 1};
  int kps[3] = {0, 0, 0};
  float* partial[3] = {nullptr, nullptr, nullptr};   // split-K fp32 partial tiles
  uint32_t* split_ctr[3] = {nullptr, nullptr, nullptr};  // split-K arrivals per tile
  int smem = 0;
  // device memory owned by the plan
  void* inter[2] = {nullptr, nullptr};
  // tile semaphores then row counters of each boundary; sems[stages - 1] (the
  // output, for desc.out_release) only when asked for
  uint32_t* sems[3] = {nullptr, nullptr, nullptr};
  size_t sem_words[3] = {0, 0, 0};
  size_t inter_bytes[2] = {0, 0};
  uint32_t* ctrl = nullptr;
  uint32_t* sched_fused = nullptr;
  int n_fused = 0;
  uint32_t* sched_stage[3] = {nullptr, nullptr, nullptr};
  int n_stage[3] = {0, 0, 0};  // entries of each stage-alone schedule (Stream-K units included)
  int workers = 0;             // clusters (or CTAs) of the plan's shape resident at once
  // Stream-K tail of the last stage (geometry in sk_*; partial tiles owned here)
  int sk_tiles = 0, sk_units = 0, sk_q = 0, sk_max_nc = 0;
  float* sk_partial = nullptr;
  // attention pieces (kv key groups each, at most kv_max per row); their
  // partial states live in partial[1], their arrivals in split_ctr[1]
  int kv = 0, kv_max = 0;
  size_t partial_bytes[3] = {0, 0, 0};
  uint32_t* delays[3] = {nullptr, nullptr, nullptr};
  unsigned long long* trace = nullptr;
  int trace_records = 0;
  int skip[3] = {-1, -1, -1};
  // TMA descriptors
  CUtensorMap maps[kMaxMaps];
  MapSlot slots[kMaxMaps];
  bool error_latched = false;
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major tensor [outer, inner] of 16-bit elements, box [box_outer, box_inner],
// 128-byte swizzle, zero fill out of bounds.
cs_status encode_2d(CUtensorMap* map, const void* ptr, int bf16, uint64_t inner, uint64_t outer, uint32_t box_inner,
                    uint32_t box_outer) {
  auto enc = get_encode();
  if (!enc) return fail(CS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable (driver too old?)");
  if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return fail(CS_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", ptr);
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(CS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu] box [%u x %u]", (int)r,
                (unsigned long long)outer, (unsigned long long)inner, box_outer, box_inner);
  return CS_OK;
}

inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Geometry shared by the host-only schedule builder and the plan.
struct Geometry {
  int stages = 0, m_tiles = 0;  // m_tiles: tile rows (tile_m each)
  int cg = 1;                   // CTAs per MMA
  int cl = 1;                   // CTAs per unit (128-row blocks per tile row)
  int m_blocks = 0;             // 128-row blocks
  int n_tiles[3] = {0, 0, 0};
  int k_iters[3] = {0, 0, 0};
  int bn[3] = {128, 128, 128};
  int splits[3] = {1, 1, 1};
  int kps[3] = {0, 0, 0};  // K-slices per split
  int lag = 1, group_m = 1, stride = 1;
  bool row_major = false;  // tiles of a group in row-major order
  bool ks_major = false;   // a split later stage's units of a group by K range first
  // Stream-K tail of the last stage: its last sk_tiles tiles in dispatch order
  // become sk_units units of sk_q consecutive K-slices each (the last shorter)
  int sk_tiles = 0, sk_units = 0, sk_q = 0, sk_max_nc = 0;
  // attention: units of tile row m cover key groups 0..m (tile_m / 128 key
  // blocks each); with kv > 0 they run as ceil((m + 1) / kv) pieces of kv groups
  int kv = 0, kv_max = 0;
};

// Smallest Stream-K share in K-slices, and the most contributors a tile may
// have (the part word holds 7 bits).
constexpr int kSkMinSlices = 8;
constexpr int kSkMaxContrib = 120;
// Allocation granule of the intermediates
constexpr size_t kInterAlloc = size_t(2) << 20;

cs_status validate(const cs_chain_desc* d) {
  if (!d) return fail(CS_ERR_INVALID_ARG, "desc is NULL");
  if (d->kind < CS_CHAIN_MLP_GELU || d->kind > CS_CHAIN_ATTN) return fail(CS_ERR_INVALID_ARG, "bad kind %d", d->kind);
  if (d->dtype != CS_F16 && d->dtype != CS_BF16) return fail(CS_ERR_INVALID_ARG, "bad dtype %d", d->dtype);
  if (d->policy < CS_SYNC_AUTO || d->policy > CS_SYNC_STREAM) return fail(CS_ERR_INVALID_ARG, "bad policy %d", d->policy);
  if (d->tuned < -1 || d->tuned > 0) return fail(CS_ERR_INVALID_ARG, "tuned=%d (0 or -1)", d->tuned);
  if (d->out_release < 0 || d->out_release > 1) return fail(CS_ERR_INVALID_ARG, "out_release=%d (0 or 1)", d->out_release);
  if (d->weight_layout != CS_WEIGHTS_KN && d->weight_layout != CS_WEIGHTS_NK)
    return fail(CS_ERR_INVALID_ARG, "bad weight_layout %d", d->weight_layout);
  if (d->M < 1 || d->M > 128 * 4095) return fail(CS_ERR_INVALID_ARG, "M=%d out of range [1, %d]", d->M, 128 * 4095);
  if (d->split_k < 0 || d->split_k > 15) return fail(CS_ERR_INVALID_ARG, "split_k=%d (0..15)", d->split_k);
  if (d->prefetch < -1 || d->prefetch > 64) return fail(CS_ERR_INVALID_ARG, "prefetch=%d (-1..64)", d->prefetch);
  if (d->raster < 0 || d->raster > 3) return fail(CS_ERR_INVALID_ARG, "raster=%d (0..3)", d->raster);
  if (d->split_k_first < 0 || d->split_k_first > 15)
    return fail(CS_ERR_INVALID_ARG, "split_k_first=%d (0..15)", d->split_k_first);
  if (d->pdl < -1 || d->pdl > 1) return fail(CS_ERR_INVALID_ARG, "pdl=%d (-1..1)", d->pdl);
  if (d->sk_tiles < -1 || d->sk_tiles > 65534) return fail(CS_ERR_INVALID_ARG, "sk_tiles=%d (-1..65534)", d->sk_tiles);
  if (d->sk_units < 0 || d->sk_units > 16383) return fail(CS_ERR_INVALID_ARG, "sk_units=%d (0..16383)", d->sk_units);
  if (d->kv_chunk < -1 || d->kv_chunk > 4095) return fail(CS_ERR_INVALID_ARG, "kv_chunk=%d (-1..4095)", d->kv_chunk);
  if (d->H < 8 || d->H % 8 != 0 || d->H > (1 << 20)) return fail(CS_ERR_INVALID_ARG, "H=%d must be a positive multiple of 8", d->H);
  if (d->F < 8 || d->F % 8 != 0 || d->F > (1 << 20)) return fail(CS_ERR_INVALID_ARG, "F=%d must be a positive multiple of 8", d->F);
  if (d->stride < 0) return fail(CS_ERR_INVALID_ARG, "stride=%d", d->stride);
  if (d->num_sms < 0) return fail(CS_ERR_INVALID_ARG, "num_sms=%d", d->num_sms);
  if (d->lag < -1) return fail(CS_ERR_INVALID_ARG, "lag=%d", d->lag);
  if (d->group_m < 0) return fail(CS_ERR_INVALID_ARG, "group_m=%d", d->group_m);
  if (d->tile_n != 0 && d->tile_n != 64 && d->tile_n != 128 && d->tile_n != 256)
    return fail(CS_ERR_INVALID_ARG, "tile_n=%d (0, 64, 128 or 256)", d->tile_n);
  if (d->tile_m != 0 && d->tile_m != 128 && d->tile_m != 256 && d->tile_m != 512)
    return fail(CS_ERR_INVALID_ARG, "tile_m=%d (0, 128, 256 or 512)", d->tile_m);
  if (d->tile_m >= 256 && (d->tile_n == 64 || d->tile_n == 128))
    return fail(CS_ERR_UNSUPPORTED, "tile_m=%d is built for 256-wide tiles only", d->tile_m);
  if (d->tile_m == 512 && !kClusterMulticast)
    return fail(CS_ERR_UNSUPPORTED, "tile_m=512 needs cluster multicast, which the replica build leaves out");
  if (d->kind == CS_CHAIN_ATTN) {
    if (d->head_dim != 128) return fail(CS_ERR_UNSUPPORTED, "head_dim=%d (only 128 is built)", d->head_dim);
    if (d->heads < 1 || d->heads * d->head_dim != d->F)
      return fail(CS_ERR_INVALID_ARG, "ATTN needs F == heads*head_dim (F=%d heads=%d)", d->F, d->heads);
    // 128 x 128 tiles on single SMs, or 256 x 256 on CTA pairs (whose attention
    // units then take two query blocks)
    if (d->tile_m == 512 || d->tile_n == 64 || (d->tile_m == 128 && d->tile_n == 256) ||
        (d->tile_m == 256 && d->tile_n == 128))
      return fail(CS_ERR_UNSUPPORTED, "the attention chain runs 128 x 128 or 256 x 256 (pair) tiles only");
  }
  return CS_OK;
}

// The desc a plan runs: the tuning table's choices for the fields left on auto
// (an entry whose choices this desc rejects is ignored), policy AUTO resolved.
cs_chain_desc resolve_desc(const cs_chain_desc* d, int num_sms, int* entry) {
  cs_chain_desc t;
  int e = cs_tune_apply(d, num_sms, &t);
  if (e >= 0) {
    char saved[sizeof(g_err)];
    std::memcpy(saved, g_err, sizeof(g_err));
    if (validate(&t) != CS_OK) e = -1, t = *d;
    std::memcpy(g_err, saved, sizeof(g_err));
  }
  if (t.policy == CS_SYNC_AUTO) t.policy = CS_SYNC_TILE;
  *entry = e;
  return t;
}

Geometry geometry(const cs_chain_desc* d, int num_sms, int workers = 0) {
  Geometry g;
  const int blocks = cdiv(d->M, cs::BM);
  // 256-wide tiles need 2/3 of the operand bytes per FLOP of 128-wide ones;
  // they pay off once the producer stage alone fills half of the grid.
  int tn = d->tile_n;
  int tm = d->tile_m;
  const bool mlp = d->kind != CS_CHAIN_ATTN;
  // Two 2-SM pairs of a 4-CTA cluster (512 x 256 tiles) fetch each weight box
  // once for both pairs (multicast).  Auto from M = 512: for SwiGLU always
  // (measured at LLaMA M=512 / 768: 76 / 104 us against 93 / 117 us with
  // 128-row tiles), for GeLU where they add no padding rows over 256-row pairs
  // (GPT-3 M=768: 199 us against 176 us with 128-row tiles).
  if (kClusterMulticast && tm == 0 && (tn == 0 || tn == 256) && mlp && blocks >= 4 &&
      (d->kind == CS_CHAIN_MLP_SWIGLU || 2 * cdiv(d->M, 512) == cdiv(d->M, 256)))
    tm = 512, tn = 256;
  if (tn == 0) tn = (2 * blocks * cdiv(d->F, 256) >= num_sms) ? 256 : 128;
  // A 2-SM pair per 256 x 256 tile halves them again (each SM loads half of B);
  // with exactly two row blocks it computes the same rows as 128-row tiles
  // (measured at M=256: GPT-3 123 -> 120 us, LLaMA 61 -> 60, stress 105 -> 94)
  if (tm == 0 && d->tile_n == 0 && mlp && blocks == 2) tm = 256, tn = 256;
  if (tm == 0) tm = (tn == 256 && mlp && blocks >= 8) ? 256 : 128;
  if (!mlp) {
    // attention: single-SM units keep S and O in TMEM next to two 128-column
    // accumulators; pair units borrow a 256-column accumulator buffer (auto
    // from M = 512, measured: M=512 134 us against 156 us; M=256 110 against 102)
    if (d->tile_m == 0) tm = blocks >= 4 ? 256 : 128;
    if (tm == 512) tm = 256;
    tn = tm == 256 ? 256 : 128;
  }
  if (tm >= 256 && tn != 256) tm = 128;
  // 512-row tiles: two 2-SM pairs of one 4-CTA cluster on consecutive 256-row
  // blocks; each weight box is fetched once and multicast to both pairs
  g.cg = tm >= 256 ? 2 : 1;
  g.cl = tm / cs::BM;
  g.m_tiles = cdiv(d->M, tm);
  g.m_blocks = g.m_tiles * g.cl;
  if (d->kind == CS_CHAIN_ATTN) {
    g.stages = 3;
    g.bn[0] = tn;
    g.n_tiles[0] = cdiv(3 * d->F, tn);
    g.k_iters[0] = cdiv(d->H, cs::BK);
    g.n_tiles[1] = d->heads;
    g.k_iters[1] = 0;
    g.bn[2] = tn;
    g.n_tiles[2] = cdiv(d->H, tn);
    g.k_iters[2] = cdiv(d->F, cs::BK);
    // Causal units grow with their row: the last rows' units lie on the
    // chain's critical path once the QKV GEMM ends.  Pieces of kv key groups
    // run them on several SMs at once, at the price of a state write and a
    // merge per piece; auto: whole rows (measured with the tensor-memory
    // accumulator, GPT-3 shard: M=1024 142 us whole against 143-147 in
    // pieces, M=2048 256 against 258-286, M=4096 543 against 553-596).  At
    // most 15 pieces per row (the unit's K-split field).
    int kv = d->kv_chunk > 0 ? d->kv_chunk : 0;
    if (kv > 0) {
      kv = std::max(kv, cdiv(g.m_tiles, 15));
      if (kv < g.m_tiles) {
        g.kv = kv;
        g.kv_max = cdiv(g.m_tiles, kv);
      }
    }
  } else {
    g.stages = 2;
    g.bn[0] = d->kind == CS_CHAIN_MLP_SWIGLU ? 128 : tn;
    g.n_tiles[0] = cdiv(d->F, g.bn[0]);
    g.k_iters[0] = cdiv(d->H, cs::BK);
    g.bn[1] = tn;
    g.n_tiles[1] = cdiv(d->H, tn);
    g.k_iters[1] = cdiv(d->F, cs::BK);
  }
  // K-splits: a stage with fewer tiles than CTAs (small M) splits K so that
  // enough SMs stream its weights (an explicit split_k: at least 8 K-slices each).
  const int capacity = num_sms / g.cl;
  for (int s = 0; s < g.stages; ++s) {
    g.splits[s] = 1;
    if (d->kind == CS_CHAIN_ATTN && s == 1) continue;  // attention units do not split
    const int tiles = g.m_tiles * g.n_tiles[s];
    // auto, more than 32 rows: at most 4 splits of at least 32 K-slices
    // (measured: finer splits make the last split's reduction and the partial
    // traffic dominate); up to 32 rows stream weights only and take up to 15
    // (measured: seven splits of a full 128-row block, stress M=128, 141 us
    // against 99 us with four)
    // an explicit count for the first stage (split_k_first) overrides split_k there
    const int want = (s == 0 && d->split_k_first > 0) ? d->split_k_first : d->split_k;
    const bool wide = want > 0 || d->M <= 32;
    const int max_sp = wide ? std::max(1, std::min(15, g.k_iters[s] / 8))
                            : std::max(1, std::min(4, g.k_iters[s] / 32));
    int sp = want;
    if (sp == 0) {
      // fewest (waves x K-slices per split): a split count that fills whole
      // waves; a larger count must win by 10 % (each split adds a partial tile
      // to write and to reduce)
      sp = 1;
      if (tiles < capacity) {
        long best = -1;
        for (int c = 1; c <= max_sp; ++c) {
          const long cost = static_cast<long>(cdiv(tiles * c, capacity)) * cdiv(g.k_iters[s], c);
          if (best < 0 || 10 * cost < 9 * best) best = cost, sp = c;
        }
      }
    }
    sp = std::min(sp, max_sp);
    sp = std::max(1, std::min(sp, 15));
    // a Stream-K tail asked for with automatic K-splits: the last stage stays
    // unsplit (its tail's units share K-slices instead)
    if (d->split_k == 0 && d->sk_tiles > 0 && s == g.stages - 1) sp = 1;
    g.kps[s] = cdiv(g.k_iters[s], sp);
    g.splits[s] = cdiv(g.k_iters[s], g.kps[s]);  // no empty split
  }
  // group_m counts tile rows.  At most 1024 rows per group; with 256-row pair
  // tiles also at least two groups, so that the lag lets the consumers of one
  // group overlap the next (measured: M=1024 pairs 0.61 -> 0.67 of peak;
  // single-SM tiles prefer one group); 512-row tiles: groups of one tile row
  // up to M = 1024 (measured at GPT-3 M=1024: 209 us with two 512-row groups,
  // 225 us with one group of 1024 rows), beyond that as below
  // GeLU chains on 512-row tiles from three tile rows: one group of up to four
  // tile rows, so every weight box is read once per 2048 rows (measured in
  // steady state: GPT-3 M=1536 322 -> 313 us, M=2048 430 -> 428 us with 680 ->
  // 442 MB of DRAM traffic per launch, stress M=1536 298 -> 286 us; SwiGLU at
  // M=2048 185 -> 196 us, so it keeps groups of two)
  g.group_m = d->group_m > 0 ? d->group_m
             : g.cl == 4   ? (g.m_tiles <= 2 ? 1 : d->kind == CS_CHAIN_MLP_GELU ? std::min(4, g.m_tiles) : 2)
             : g.cg == 2   ? std::max(1, std::min(4, g.m_tiles / 2))
                           : 8;
  g.row_major = d->raster == 2;
  g.ks_major = d->raster == 3;
  if (g.group_m > g.m_tiles) g.group_m = g.m_tiles;
  const int groups = cdiv(g.m_tiles, g.group_m);
  g.lag = d->lag >= 0 ? d->lag : 1;
  if (g.lag > groups) g.lag = groups;
  g.stride = d->stride > 0 ? d->stride : (d->kind == CS_CHAIN_ATTN ? d->heads : 4);
  // Stream-K tail: the last stage's trailing tiles (at most those of the last
  // row group, all listed at the schedule's end) shared out in equal K-ranges
  const int fs = g.stages - 1;
  if (d->sk_tiles > 0 && g.splits[fs] == 1 && g.k_iters[fs] >= 2) {
    const int last_rows = g.m_tiles - (groups - 1) * g.group_m;
    const int tiles = std::min(d->sk_tiles, last_rows * g.n_tiles[fs]);
    const long long K = g.k_iters[fs];
    const long long work = static_cast<long long>(tiles) * K;
    const int units = d->sk_units > 0 ? d->sk_units : (workers > 0 ? workers : capacity);
    long long q = (work + units - 1) / units;
    q = std::max<long long>(q, std::min<long long>(kSkMinSlices, K));
    q = std::max<long long>(q, (K + kSkMaxContrib - 2) / (kSkMaxContrib - 1));
    g.sk_tiles = tiles;
    g.sk_q = static_cast<int>(q);
    g.sk_units = static_cast<int>((work + q - 1) / q);
    g.sk_max_nc = 0;
    for (int j = 0; j < tiles; ++j)
      g.sk_max_nc = std::max(g.sk_max_nc, static_cast<int>(((j + 1) * K - 1) / q - (j * K) / q + 1));
  }
  return g;
}

// Dispatch order (closed form in cs_sched.cuh, shared with the device-side
// builder of the allocation-free forward): row tiles in groups of group_m; at
// step t, stage s lists the units of group t - s*lag, so every producer unit a
// consumer waits on is listed before it and an in-order dispatcher cannot
// deadlock.
cs::SchedGeo sched_geo(const Geometry& g) {
  cs::SchedGeo sg;
  sg.stages = g.stages;
  sg.m_tiles = g.m_tiles;
  sg.group_m = g.group_m;
  sg.lag = g.lag;
  sg.row_major = g.row_major ? 1 : 0;
  sg.ks_major = g.ks_major ? 1 : 0;
  for (int s = 0; s < 3; ++s) {
    sg.n_tiles[s] = g.n_tiles[s];
    sg.splits[s] = g.splits[s];
  }
  if (g.stages == 3) sg.kv[1] = g.kv;
  return sg;
}

// A schedule as uploaded: n_units dispatch entries, then (with a Stream-K
// tail) the unit encodings of the sk_tiles tiles the Stream-K units share.
struct Sched {
  std::vector<uint32_t> v;
  int n_units = 0;
};

// The last g.sk_tiles entries (the last stage's trailing tiles) become the
// Stream-K table; Stream-K units (K-split field 15, unit index in the column
// field) take their place.
Sched with_stream_k(const Geometry& g, std::vector<uint32_t> v, bool last_stage) {
  Sched r;
  if (!last_stage || g.sk_units == 0 || static_cast<int>(v.size()) < g.sk_tiles) {
    r.n_units = static_cast<int>(v.size());
    r.v = std::move(v);
    return r;
  }
  const size_t keep = v.size() - static_cast<size_t>(g.sk_tiles);
  std::vector<uint32_t> table(v.begin() + static_cast<long>(keep), v.end());
  v.resize(keep);
  for (int u = 0; u < g.sk_units; ++u) v.push_back(cs::sched_enc(g.stages - 1, 0, u, cs::SK_KS));
  r.n_units = static_cast<int>(v.size());
  v.insert(v.end(), table.begin(), table.end());
  r.v = std::move(v);
  return r;
}

Sched build_fused(const Geometry& g) {
  const cs::SchedGeo sg = sched_geo(g);
  std::vector<uint32_t> v(static_cast<size_t>(cs::sched_fused_count(sg)));
  for (size_t i = 0; i < v.size(); ++i) v[i] = cs::sched_fused_entry(sg, static_cast<long long>(i));
  return with_stream_k(g, std::move(v), true);
}

// One stage alone (two-kernel control, standalone timings): same grouping, and
// the same Stream-K tail on the last stage (so its bits equal the fused chain's).
Sched build_stage(const Geometry& g, int s) {
  const cs::SchedGeo sg = sched_geo(g);
  std::vector<uint32_t> v(static_cast<size_t>(cs::sched_stage_count(sg, s)));
  for (size_t i = 0; i < v.size(); ++i) v[i] = cs::sched_stage_entry(sg, s, static_cast<long long>(i));
  return with_stream_k(g, std::move(v), s == g.stages - 1);
}

// Everything a plan takes from its geometry: tile counts, K-splits, the kernel
// configuration (ring depth and stage size) and its shared memory.  The grid
// is rounded down to whole clusters.
void shape_plan(cs_chain_s* p, const Geometry& g, int kind, int M) {
  p->m_tiles = g.m_blocks;
  p->m_units = g.m_tiles;
  p->m_blocks = g.m_blocks;
  p->cg = g.cg;
  p->cl = g.cl;
  p->stages = g.stages;
  for (int i = 0; i < 3; ++i) {
    p->n_tiles[i] = g.n_tiles[i];
    p->k_iters[i] = g.k_iters[i];
    p->units[i] = g.m_blocks * g.n_tiles[i];
    p->sched_units[i] = i < g.stages ? static_cast<int>(cs::sched_stage_count(sched_geo(g), i)) : 0;
    p->splits[i] = g.splits[i];
    p->kps[i] = g.kps[i];
    p->bn[i] = g.bn[i];
  }
  p->lag = g.lag;
  p->group_m = g.group_m;
  p->raster = g.row_major ? 2 : g.ks_major ? 3 : 1;
  p->stride = g.stride;
  p->sk_tiles = g.sk_tiles;
  p->sk_units = g.sk_units;
  p->sk_q = g.sk_q;
  p->sk_max_nc = g.sk_max_nc;
  p->kv = g.kv;
  p->kv_max = g.kv_max;
  const bool wide_b = kind == CS_CHAIN_MLP_SWIGLU || g.bn[0] == 256 || g.bn[1] == 256 || g.bn[2] == 256;
  p->cfg_s = (g.cg == 1 && kind != CS_CHAIN_ATTN && M <= 32) ? (M <= 8 ? 1 : 3) + (wide_b ? 1 : 0) : 0;
  p->cfg_b = g.cg == 1 && !p->cfg_s && wide_b;
  p->smem = p->cfg_s == 1 ? smem_bytes_for<NS_S, SB_S>()
            : p->cfg_s == 2 ? smem_bytes_for<NS_T, SB_T>()
            : p->cfg_s == 3 ? smem_bytes_for<NS_U, SB_U>()
            : p->cfg_s == 4 ? smem_bytes_for<NS_V, SB_V>()
            : p->cfg_b      ? smem_bytes_for<NS_B, SB_B>()
                            : smem_bytes_for<NS_A, SB_A>();
  p->num_sms = p->num_sms / g.cl * g.cl;
}

// The geometry fields of cs_chain_info (no device pointers).
void info_geometry(const cs_chain_s* p, int n_fused, cs_chain_info* info) {
  std::memset(info, 0, sizeof(*info));
  info->stages = p->stages;
  info->m_tiles = p->m_tiles;
  for (int i = 0; i < 3; ++i) {
    info->n_tiles[i] = p->n_tiles[i];
    info->units[i] = p->units[i];
    info->tile_n[i] = p->bn[i];
    info->sched_units[i] = p->sched_units[i];
    info->split_k[i] = p->splits[i];
  }
  info->n_units = n_fused;
  info->num_sms = p->num_sms;
  info->smem_bytes = p->smem;
  info->lag = p->lag;
  info->group_m = p->group_m;
  info->tile_m = cs::BM * p->cl;
  info->stride = p->stride;
  info->policy = p->d.policy;
  info->tuned_entry = p->tuned_entry;
  info->sk_tiles = p->sk_tiles;
  info->sk_units = p->sk_units;
  info->sk_q = p->sk_q;
  info->workers = p->workers > 0 ? p->workers : p->num_sms / p->cl;
  info->kv_chunk = p->kv;
  info->raster = p->raster;
}

int device_sms(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  *out = v;
  return dev;
}

template <int NS, int SB, int CG, bool ATTN, int CL = CG, int AR = cs::BM>
cs_status set_smem_attr() {
  static cudaError_t once = cudaFuncSetAttribute(cs::cs_chain_kernel<NS, SB, CG, ATTN, CL, AR>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes_for<NS, SB>());
  if (once != cudaSuccess) return fail(CS_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(once));
  return CS_OK;
}

void free_plan(cs_chain_s* p) {
  if (!p) return;
  for (auto& b : p->inter) if (b) cudaFree(b);
  for (auto& b : p->sems) if (b) cudaFree(b);
  if (p->ctrl) cudaFree(p->ctrl);
  if (p->sched_fused) cudaFree(p->sched_fused);
  for (auto& b : p->sched_stage) if (b) cudaFree(b);
  for (auto& b : p->delays) if (b) cudaFree(b);
  if (p->trace) cudaFree(p->trace);
  for (auto& b : p->partial) if (b) cudaFree(b);
  for (auto& b : p->split_ctr) if (b) cudaFree(b);
  if (p->sk_partial) cudaFree(p->sk_partial);
  for (auto& b : p->host_x) if (b) cudaFree(b);
  for (auto& b : p->host_y) if (b) cudaFree(b);
  for (cudaEvent_t* evs : {p->ev_x, p->ev_k, p->ev_y})
    for (int i = 0; i < 2; ++i) if (evs[i]) cudaEventDestroy(evs[i]);
  if (p->s_h2d) cudaStreamDestroy(p->s_h2d);
  if (p->s_d2h) cudaStreamDestroy(p->s_d2h);
  delete p;
}

template <typename T>
cs_status upload(T** dst, const std::vector<T>& v) {
  if (v.empty()) {
    *dst = nullptr;
    return CS_OK;
  }
  if (cudaMalloc(reinterpret_cast<void**>(dst), v.size() * sizeof(T)) != cudaSuccess)
    return fail(CS_ERR_OOM, "cudaMalloc(%zu) failed", v.size() * sizeof(T));
  CS_CUDA(cudaMemcpy(*dst, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice));
  return CS_OK;
}

// Map indices (MLP): 0 X, 1 W1/Wg, 2 Wu, 3 H store, 4 H load, 5 W2, 6 Y store.
enum { MAP_X = 0, MAP_W1 = 1, MAP_WU = 2, MAP_HST = 3, MAP_HLD = 4, MAP_W2 = 5, MAP_Y = 6 };

// Encode a weight map: math shape [K, N].  KN storage: row-major [K, N], boxes of
// 64 N x 64 K.  NK storage: row-major [N, K], boxes of 64 K x box_n N rows (the
// columns of a tile one CTA loads).
cs_status encode_weight(cs_chain_s* p, int slot, const void* ptr, int K, int N, int box_n) {
  if (p->slots[slot].valid && p->slots[slot].ptr == ptr) return CS_OK;
  const int bf16 = p->d.dtype == CS_BF16;
  cs_status s = p->d.weight_layout == CS_WEIGHTS_KN ? encode_2d(&p->maps[slot], ptr, bf16, N, K, 64, 64)
                                                     : encode_2d(&p->maps[slot], ptr, bf16, K, N, 64, box_n);
  if (s != CS_OK) return s;
  p->slots[slot].ptr = ptr;
  p->slots[slot].valid = true;
  return CS_OK;
}

// Activation-side map: row-major [rows, cols]; box 64 cols x (128 rows for loads / 32 for stores).
cs_status encode_act(cs_chain_s* p, int slot, const void* ptr, int rows, int cols, bool store, int load_rows = 128) {
  if (p->slots[slot].valid && p->slots[slot].ptr == ptr) return CS_OK;
  cs_status s = encode_2d(&p->maps[slot], ptr, p->d.dtype == CS_BF16, cols, rows, 64, store ? 32 : load_rows);
  if (s != CS_OK) return s;
  p->slots[slot].ptr = ptr;
  p->slots[slot].valid = true;
  return CS_OK;
}

// Two-kernel control: the launch of the next stage records its units after
// those of stage `done` in the trace buffer (each launch counts its dispatch
// indices from 0).
void next_trace_segment(const cs_chain_s* p, cs::KParams& kp, int done) {
  if (!kp.trace) return;
  const int recs = p->n_stage[done] * p->cl;
  kp.trace += static_cast<size_t>(recs) * cs::TRACE_WORDS;
  kp.trace_records -= recs;
}

int wait_kind(const cs_chain_s* p) {
  return p->d.policy == CS_SYNC_TILE ? cs::WAIT_TILE
         : p->d.policy == CS_SYNC_ROW ? cs::WAIT_ROW
         : p->d.policy == CS_SYNC_STRIDED ? cs::WAIT_STRIDED
                                          : cs::WAIT_NONE;
}

void fill_split(const cs_chain_s* p, int st, cs::StageP& s) {
  s.splits = p->splits[st];
  s.kps = p->kps[st] > 0 ? p->kps[st] : p->k_iters[st];
  s.m_blocks = p->m_blocks;
  s.partial = p->partial[st];
  s.split_ctr = p->split_ctr[st];
  if (st == p->stages - 1 && p->sk_units > 0) {
    s.sk_tiles = p->sk_tiles;
    s.sk_units = p->sk_units;
    s.sk_q = p->sk_q;
    s.sk_max_nc = p->sk_max_nc;
    s.sk_partial = p->sk_partial;
  }
}

void fill_common(const cs_chain_s* p, cs::KParams& kp) {
  std::memcpy(kp.maps, p->maps, sizeof(kp.maps));
  kp.ctrl = p->ctrl;
  kp.timeout_ns = p->d.spin_timeout_ns ? p->d.spin_timeout_ns : kDefaultTimeoutNs;
  kp.watchdog_ns = kp.timeout_ns * 4 > 4000000000ull ? kp.timeout_ns * 4 : 4000000000ull;
  kp.bf16 = p->d.dtype == CS_BF16;
  kp.trace = p->trace;
  kp.trace_records = p->trace_records;
  // measured: extra L2 prefetch requests slow the loads down, so auto = off
  kp.pf_dist = p->d.prefetch <= 0 ? 0 : p->d.prefetch;
}

// Raw pointers and strides of a GEMM stage's operands for the L2 prefetch.
// Weight math shape [K, N]: KN storage has K rows of N, NK storage N rows of K.
void fill_prefetch(const cs_chain_s* p, cs::StageP& s, const void* w, const void* w2, int K, int N, const void* a,
                   int a_rows, int a_cols) {
  const bool kn = p->d.weight_layout == CS_WEIGHTS_KN;
  s.pf_b = static_cast<const char*>(w);
  s.pf_b2 = static_cast<const char*>(w2);
  s.pf_ldb = static_cast<long long>(kn ? N : K) * 2;
  s.pf_brows = kn ? K : N;
  s.pf_a = static_cast<const char*>(a);
  s.pf_lda = static_cast<long long>(a_cols) * 2;
  s.pf_arows = a_rows;
}

void fill_mlp_stages(const cs_chain_s* p, const cs_mlp_args* a, cs::KParams& kp) {
  const bool swiglu = p->d.kind == CS_CHAIN_MLP_SWIGLU;
  const int b_major = p->d.weight_layout == CS_WEIGHTS_KN ? 1 : 0;
  const int wait = wait_kind(p);
  cs::StageP& s0 = kp.st[0];
  std::memset(&s0, 0, sizeof(s0));
  s0.kind = cs::STAGE_GEMM;
  s0.epi = swiglu ? cs::EPI_SWIGLU : cs::EPI_BIAS_GELU;
  s0.m_tiles = p->m_tiles;
  s0.n_tiles = p->n_tiles[0];
  s0.k_iters = p->k_iters[0];
  s0.n_extent = p->d.F;
  s0.m_extent = p->d.M;
  s0.bn = p->bn[0];
  s0.mma_n = swiglu ? 256 : p->bn[0];
  s0.b_major = b_major;
  s0.map_a = MAP_X;
  s0.map_b = MAP_W1;
  s0.map_b2 = swiglu ? MAP_WU : -1;
  s0.map_out = MAP_HST;
  s0.b_bytes = (swiglu ? 2 : 1) * (p->bn[0] / p->cg) * cs::BK * 2;
  s0.bias_f16 = reinterpret_cast<const __half*>(a ? a->b1 : nullptr);
  s0.bias_bf16 = reinterpret_cast<const __nv_bfloat16*>(a ? a->b1 : nullptr);
  s0.wait = cs::WAIT_NONE;
  s0.rel_tile = p->sems[0];
  s0.rel_row = p->sems[0] + static_cast<size_t>(p->m_blocks) * p->n_tiles[0];
  s0.delay_ns = p->delays[0];
  s0.skip_unit = p->skip[0];

  cs::StageP& s1 = kp.st[1];
  std::memset(&s1, 0, sizeof(s1));
  s1.kind = cs::STAGE_GEMM;
  s1.epi = cs::EPI_NONE;
  s1.m_tiles = p->m_tiles;
  s1.n_tiles = p->n_tiles[1];
  s1.k_iters = p->k_iters[1];
  s1.n_extent = p->d.H;
  s1.m_extent = p->d.M;
  s1.bn = p->bn[1];
  s1.mma_n = p->bn[1];
  s1.b_major = b_major;
  s1.map_a = MAP_HLD;
  s1.map_b = MAP_W2;
  s1.map_b2 = -1;
  s1.map_out = MAP_Y;
  s1.b_bytes = (p->bn[1] / p->cg) * cs::BK * 2;
  s1.wait = wait;
  s1.dep_tile = p->sems[0];
  s1.dep_row = p->sems[0] + static_cast<size_t>(p->m_blocks) * p->n_tiles[0];
  s1.dep_ntiles = p->n_tiles[0];
  s1.dep_bn = p->bn[0];
  s1.stride = p->stride;
  // the output's own semaphores when the plan releases Y (desc.out_release)
  s1.rel_tile = p->sems[1];
  s1.rel_row = p->sems[1] ? p->sems[1] + p->sem_words[1] : nullptr;
  s1.skip_unit = -1;
  fill_split(p, 0, s0);
  fill_split(p, 1, s1);
  if (a) {
    fill_prefetch(p, s0, swiglu ? a->Wg : a->W1, swiglu ? a->Wu : nullptr, p->d.H, p->d.F, a->X, p->d.M, p->d.H);
    fill_prefetch(p, s1, a->W2, nullptr, p->d.F, p->d.H, nullptr, 0, 0);
    // raw outputs for the plain-store epilogue of small split tiles
    s0.out_ptr = p->inter[0];
    s0.out_ld = p->d.F;
    s1.out_ptr = a->Y;
    s1.out_ld = p->d.H;
  }
  kp.acc_stride = (s0.mma_n > 128 || s1.mma_n > 128) ? 256 : 128;
}

// The kernel instantiation a plan runs (its shared-memory size set once).
cs_status kernel_for(const cs_chain_s* p, const void** fn) {
  cs_status s;
#define CS_KERNEL(...)                                                                  \
  do {                                                                                  \
    if ((s = set_smem_attr<__VA_ARGS__>()) != CS_OK) return s;                           \
    *fn = reinterpret_cast<const void*>(cs::cs_chain_kernel<__VA_ARGS__>);              \
    return CS_OK;                                                                       \
  } while (0)
  if (p->d.kind == CS_CHAIN_ATTN && p->cg == 2) CS_KERNEL(NS_A, SB_A, 2, true);
  if (p->d.kind == CS_CHAIN_ATTN) CS_KERNEL(NS_A, SB_A, 1, true);
#ifndef CS_NO_CLUSTER_MULTICAST
  if (p->cl == 4) CS_KERNEL(NS_A, SB_A, 2, false, 4);
#endif
  if (p->cg == 2) CS_KERNEL(NS_A, SB_A, 2, false);
  if (p->cfg_s == 1) CS_KERNEL(NS_S, SB_S, 1, false, 1, 8);
  if (p->cfg_s == 2) CS_KERNEL(NS_T, SB_T, 1, false, 1, 8);
  if (p->cfg_s == 3) CS_KERNEL(NS_U, SB_U, 1, false, 1, 32);
  if (p->cfg_s == 4) CS_KERNEL(NS_V, SB_V, 1, false, 1, 32);
  if (p->cfg_b) CS_KERNEL(NS_B, SB_B, 1, false);
  CS_KERNEL(NS_A, SB_A, 1, false);
#undef CS_KERNEL
}

// Rows of the A operand per pipeline stage (and of the activation load boxes):
// 8 up to 8 rows, 32 up to 32, else the full 128-row block.
int a_rows(const cs_chain_s* p) { return p->cfg_s == 1 || p->cfg_s == 2 ? 8 : p->cfg_s ? 32 : cs::BM; }

// Threads per CTA: the attention instantiations run two epilogue warps per TMEM
// lane quadrant.
unsigned block_threads(const cs_chain_s* p) {
  return static_cast<unsigned>(p->d.kind == CS_CHAIN_ATTN ? cs::Roles<true>::THREADS : cs::Roles<false>::THREADS);
}

// Clusters of the plan's shape that can be resident at once: a GPC whose SM
// count is not a multiple of the cluster size leaves SMs idle (on a 152-SM
// GB300, 36 clusters of 4 CTAs, 144 SMs).
cs_status resident_workers(const cs_chain_s* p, int* workers) {
  *workers = p->num_sms / p->cl;
  if (p->cl == 1) return CS_OK;
  const void* fn = nullptr;
  cs_status s = kernel_for(p, &fn);
  if (s != CS_OK) return s;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p->num_sms);
  cfg.blockDim = dim3(block_threads(p));
  cfg.dynamicSmemBytes = p->smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = static_cast<unsigned>(p->cl);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  CS_CUDA(cudaOccupancyMaxActiveClusters(&n, fn, &cfg));
  if (n >= 1 && n < *workers) *workers = n;
  return CS_OK;
}

cs_status launch(cs_chain_s* p, cs::KParams& kp, const uint32_t* sched, int n_units, cudaStream_t stream) {
  kp.sched = sched;
  kp.n_units = n_units;
  // a schedule with Stream-K units is followed by the table of their tiles
  kp.st[p->stages - 1].sk_tile = sched + n_units;
  // one CTA per SM, clusters of cl CTAs per unit: as many clusters as can be
  // resident at once, and no more than units
  int grid = p->workers > 0 ? p->workers : p->num_sms / p->cl;
  if (grid > n_units) grid = n_units;
  if (grid < 1) grid = 1;
  grid *= p->cl;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block_threads(p));
  cfg.dynamicSmemBytes = p->smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (p->cl > 1) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = static_cast<unsigned>(p->cl);
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  if (p->d.pdl >= 0) {
    // the kernel waits for the preceding grid (griddepcontrol.wait) before it
    // touches global memory, so it may be scheduled while that grid drains
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  cfg.attrs = n_attr ? attr : nullptr;
  cfg.numAttrs = n_attr;
  const void* fn = nullptr;
  cs_status s = kernel_for(p, &fn);
  if (s != CS_OK) return s;
  void* args[] = {&kp};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return fail(CS_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  return CS_OK;
}

// Map indices (ATTN): 0 X, 1 Wqkv, 2 QKV store, 3 QKV load, 4 O store, 5 O load, 6 Wo, 7 Y store.
// 8 K half: QKV loads of 64-row boxes (half a key block, attention on CTA pairs).
enum { AMAP_X = 0, AMAP_WQKV = 1, AMAP_QKVST = 2, AMAP_QKVLD = 3, AMAP_OST = 4, AMAP_OLD = 5, AMAP_WO = 6, AMAP_Y = 7,
       AMAP_K64 = 8 };

void fill_attn_stages(const cs_chain_s* p, cs::KParams& kp) {
  const int b_major = p->d.weight_layout == CS_WEIGHTS_KN ? 1 : 0;
  const int F = p->d.F, H = p->d.H, M = p->d.M;
  uint32_t* rows0 = p->sems[0] + static_cast<size_t>(p->m_blocks) * p->n_tiles[0];
  uint32_t* rows1 = p->sems[1] + static_cast<size_t>(p->m_blocks) * p->n_tiles[1];
  // stage 0: QKV = X Wqkv
  cs::StageP& s0 = kp.st[0];
  std::memset(&s0, 0, sizeof(s0));
  s0.kind = cs::STAGE_GEMM;
  s0.epi = cs::EPI_NONE;
  s0.m_tiles = p->m_units;
  s0.n_tiles = p->n_tiles[0];
  s0.k_iters = p->k_iters[0];
  s0.n_extent = 3 * F;
  s0.m_extent = M;
  s0.bn = p->bn[0];
  s0.mma_n = p->bn[0];
  s0.b_major = b_major;
  s0.map_a = AMAP_X;
  s0.map_b = AMAP_WQKV;
  s0.map_b2 = -1;
  s0.map_out = AMAP_QKVST;
  s0.b_bytes = (p->bn[0] / p->cg) * cs::BK * 2;
  s0.wait = cs::WAIT_NONE;
  s0.rel_tile = p->sems[0];
  s0.rel_row = rows0;
  s0.delay_ns = p->delays[0];
  s0.skip_unit = p->skip[0];
  // stage 1: causal attention, one unit per (128-query block, head)
  cs::StageP& s1 = kp.st[1];
  std::memset(&s1, 0, sizeof(s1));
  s1.kind = cs::STAGE_ATTN;
  s1.m_tiles = p->m_units;
  s1.n_tiles = p->n_tiles[1];
  s1.n_extent = F;
  s1.m_extent = M;
  s1.bn = 128;
  s1.map_a = AMAP_QKVLD;
  s1.map_k = AMAP_K64;
  s1.map_b = -1;
  s1.map_b2 = -1;
  s1.map_out = AMAP_OST;
  s1.wait = wait_kind(p);
  s1.dep_tile = p->sems[0];
  s1.dep_row = rows0;
  s1.dep_ntiles = p->n_tiles[0];
  s1.dep_bn = p->bn[0];
  s1.stride = p->stride;
  s1.rel_tile = p->sems[1];
  s1.rel_row = rows1;
  s1.delay_ns = p->delays[1];
  s1.skip_unit = p->skip[1];
  s1.heads = p->d.heads;
  s1.softmax_scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(p->d.head_dim)));
  // stage 2: Y = O Wo
  cs::StageP& s2 = kp.st[2];
  std::memset(&s2, 0, sizeof(s2));
  s2.kind = cs::STAGE_GEMM;
  s2.epi = cs::EPI_NONE;
  s2.m_tiles = p->m_units;
  s2.n_tiles = p->n_tiles[2];
  s2.k_iters = p->k_iters[2];
  s2.n_extent = H;
  s2.m_extent = M;
  s2.bn = p->bn[2];
  s2.mma_n = p->bn[2];
  s2.b_major = b_major;
  s2.map_a = AMAP_OLD;
  s2.map_b = AMAP_WO;
  s2.map_b2 = -1;
  s2.map_out = AMAP_Y;
  s2.b_bytes = (p->bn[2] / p->cg) * cs::BK * 2;
  s2.wait = wait_kind(p);
  s2.dep_tile = p->sems[1];
  s2.dep_row = rows1;
  s2.dep_ntiles = p->n_tiles[1];
  s2.dep_bn = 128;
  s2.stride = p->stride;
  s2.rel_tile = p->sems[2];
  s2.rel_row = p->sems[2] ? p->sems[2] + p->sem_words[2] : nullptr;
  s2.skip_unit = -1;
  fill_split(p, 0, s0);
  fill_split(p, 1, s1);
  fill_split(p, 2, s2);
  s1.kv_chunk = p->kv;
  s1.kv_max = p->kv_max;
  // pairs: 256-column buffers, which attention units borrow for S and O
  kp.acc_stride = p->cg == 2 ? 256 : 128;
}

void fill_attn_prefetch(const cs_chain_s* p, const cs_attn_args* a, cs::KParams& kp) {
  fill_prefetch(p, kp.st[0], a->Wqkv, nullptr, p->d.H, 3 * p->d.F, a->X, p->d.M, p->d.H);
  fill_prefetch(p, kp.st[2], a->Wo, nullptr, p->d.F, p->d.H, nullptr, 0, 0);
  // raw outputs for the plain-store epilogue of small split tiles
  kp.st[0].out_ptr = p->inter[0];
  kp.st[0].out_ld = 3 * p->d.F;
  kp.st[2].out_ptr = a->Y;
  kp.st[2].out_ld = p->d.H;
}

cs_status bind_attn(cs_chain_s* p, const cs_attn_args* a) {
  if (!a) return fail(CS_ERR_INVALID_ARG, "args is NULL");
  if (!a->X || !a->Wqkv || !a->Wo || !a->Y) return fail(CS_ERR_INVALID_ARG, "X, Wqkv, Wo and Y are required");
  const int M = p->d.M, H = p->d.H, F = p->d.F;
  cs_status s;
  if ((s = encode_act(p, AMAP_X, a->X, M, H, false)) != CS_OK) return s;
  if ((s = encode_weight(p, AMAP_WQKV, a->Wqkv, H, 3 * F, p->bn[0] / p->cg)) != CS_OK) return s;
  if ((s = encode_weight(p, AMAP_WO, a->Wo, F, H, p->bn[2] / p->cg)) != CS_OK) return s;
  if ((s = encode_act(p, AMAP_Y, a->Y, M, H, true)) != CS_OK) return s;
  return CS_OK;
}

cs_status bind_mlp(cs_chain_s* p, const cs_mlp_args* a) {
  if (!a) return fail(CS_ERR_INVALID_ARG, "args is NULL");
  const bool swiglu = p->d.kind == CS_CHAIN_MLP_SWIGLU;
  if (!a->X || !a->W2 || !a->Y) return fail(CS_ERR_INVALID_ARG, "X, W2 and Y are required");
  if (swiglu ? (!a->Wg || !a->Wu) : (!a->W1 || !a->b1))
    return fail(CS_ERR_INVALID_ARG, swiglu ? "Wg and Wu are required" : "W1 and b1 are required");
  if (!swiglu && reinterpret_cast<uintptr_t>(a->b1) % 16 != 0) return fail(CS_ERR_INVALID_ARG, "b1 is not 16-byte aligned");
  const int M = p->d.M, H = p->d.H, F = p->d.F;
  cs_status s;
  if ((s = encode_act(p, MAP_X, a->X, M, H, false, a_rows(p))) != CS_OK) return s;
  // [N, K] weights: a box holds the B columns one CTA fetches (with 4-CTA
  // clusters, half of its pair share; the other half comes by multicast).  A
  // gate|up pair gives each CTA all bn rows of one of the two operands.
  const int split_b = p->cl == 4 ? 2 : 1;
  const int box0 = (swiglu ? p->bn[0] : p->bn[0] / p->cg) / split_b;
  if ((s = encode_weight(p, MAP_W1, swiglu ? a->Wg : a->W1, H, F, box0)) != CS_OK) return s;
  if (swiglu && (s = encode_weight(p, MAP_WU, a->Wu, H, F, box0)) != CS_OK) return s;
  if ((s = encode_weight(p, MAP_W2, a->W2, F, H, p->bn[1] / p->cg / split_b)) != CS_OK) return s;
  if ((s = encode_act(p, MAP_Y, a->Y, M, H, true)) != CS_OK) return s;
  return CS_OK;
}

}  // namespace

extern "C" {

int cs_abi_version(void) { return CS_ABI_VERSION; }

const char* cs_last_error_string(void) { return g_err; }

cs_status cs_chain_desc_init(cs_chain_desc* d) {
  if (!d) return fail(CS_ERR_INVALID_ARG, "desc is NULL");
  std::memset(d, 0, sizeof(*d));
  d->kind = CS_CHAIN_MLP_GELU;
  d->dtype = CS_F16;
  d->policy = CS_SYNC_TILE;
  d->weight_layout = CS_WEIGHTS_KN;
  d->heads = 12;
  d->head_dim = 128;
  d->lag = -1;
  d->group_m = 0;
  d->tile_n = 0;
  d->tile_m = 0;
  d->split_k = 0;
  d->prefetch = 0;
  d->raster = 0;
  d->pdl = 0;
  d->tuned = 0;
  d->out_release = 0;
  return CS_OK;
}

cs_status cs_schedule_build(const cs_chain_desc* desc, int num_sms, uint32_t* units, size_t cap, size_t* n_out) {
  cs_status s = validate(desc);
  if (s != CS_OK) return s;
  if (num_sms < 1) return fail(CS_ERR_INVALID_ARG, "num_sms=%d", num_sms);
  if (!n_out) return fail(CS_ERR_INVALID_ARG, "n_out is NULL");
  if (cap > 0 && !units) return fail(CS_ERR_INVALID_ARG, "units is NULL");
  int entry = -1;
  const cs_chain_desc rd = resolve_desc(desc, num_sms, &entry);
  Geometry g = geometry(&rd, num_sms);
  const Sched f = build_fused(g);
  *n_out = static_cast<size_t>(f.n_units);
  for (size_t i = 0; i < *n_out && i < cap; ++i) units[i] = f.v[i];
  return CS_OK;
}

cs_status cs_chain_plan(const cs_chain_desc* desc, cs_chain_t* out) {
  if (!out) return fail(CS_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  cs_status s = validate(desc);
  if (s != CS_OK) return s;
  int sms = 0;
  const int dev = device_sms(&sms);
  if (dev < 0) return fail(CS_ERR_CUDA, "no CUDA device available");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major * 10 + minor != 103)
    return fail(CS_ERR_UNSUPPORTED, "device is sm_%d%d; this library is built for sm_103a only", major, minor);

  cs_chain_s* p = new (std::nothrow) cs_chain_s();
  if (!p) return fail(CS_ERR_OOM, "host allocation failed");
  p->device = dev;
  const int grid_sms = desc->num_sms > 0 && desc->num_sms < sms ? desc->num_sms : sms;
  p->num_sms = grid_sms;
  p->d = resolve_desc(desc, p->num_sms, &p->tuned_entry);
  Geometry g = geometry(&p->d, p->num_sms);
  shape_plan(p, g, desc->kind, desc->M);
  if ((s = resident_workers(p, &p->workers)) != CS_OK) {
    delete p;
    return s;
  }
  if (g.sk_units > 0 && p->d.sk_units == 0 && p->workers != p->num_sms / g.cl) {
    // one Stream-K unit per resident worker
    p->num_sms = grid_sms;
    g = geometry(&p->d, grid_sms, p->workers);
    shape_plan(p, g, desc->kind, desc->M);
  }

  auto bail = [&](cs_status st) {
    free_plan(p);
    return st;
  };
  const size_t esz = 2;
  // intermediate H [M, F]
  const bool attn = desc->kind == CS_CHAIN_ATTN;
  // intermediates: H [M, F] (MLP); QKV [M, 3F] and O [M, F] (attention)
  p->inter_bytes[0] = static_cast<size_t>(desc->M) * (attn ? 3 : 1) * desc->F * esz;
  p->inter_bytes[1] = attn ? static_cast<size_t>(desc->M) * desc->F * esz : 0;
  // Each intermediate gets an allocation of whole 2 MB: a small one shares the
  // driver's small-allocation pages, where the chain's time at small M depends
  // on where it lands (measured, 16 identical plans of the GPT-3 attention
  // chain at M=16: 51.8-65.8 us, 51.8-52.9 us with whole 2 MB; LLaMA M=16 mean
  // 49.8 -> 47.0 us).
  for (int b = 0; b < 2; ++b)
    if (p->inter_bytes[b] &&
        cudaMalloc(&p->inter[b], (p->inter_bytes[b] + kInterAlloc - 1) / kInterAlloc * kInterAlloc) != cudaSuccess)
      return bail(fail(CS_ERR_OOM, "cudaMalloc of the intermediate failed"));
  for (int b = 0; b < g.stages - (desc->out_release ? 0 : 1); ++b) {
    p->sem_words[b] = static_cast<size_t>(g.m_blocks) * g.n_tiles[b];
    const size_t words = p->sem_words[b] + g.m_blocks;
    if (cudaMalloc(reinterpret_cast<void**>(&p->sems[b]), words * 4) != cudaSuccess)
      return bail(fail(CS_ERR_OOM, "cudaMalloc of semaphores failed"));
    if (cudaMemset(p->sems[b], 0, words * 4) != cudaSuccess) return bail(fail(CS_ERR_CUDA, "cudaMemset failed"));
  }
  if (cudaMalloc(reinterpret_cast<void**>(&p->ctrl), cs::CTRL_WORDS * 4) != cudaSuccess)
    return bail(fail(CS_ERR_OOM, "cudaMalloc of the control block failed"));
  for (int st = 0; st < g.stages; ++st) {
    const bool sk = st == g.stages - 1 && g.sk_units > 0;
    if (sk) {
      // Stream-K partial tiles: [sk_tiles][sk_max_nc][CTAs per unit][128][tile_n]
      const size_t pf = static_cast<size_t>(g.sk_tiles) * g.sk_max_nc * g.cl * cs::BM * g.bn[st];
      const size_t words = static_cast<size_t>(g.m_blocks) * g.n_tiles[st];
      if (cudaMalloc(reinterpret_cast<void**>(&p->sk_partial), pf * 4) != cudaSuccess ||
          cudaMalloc(reinterpret_cast<void**>(&p->split_ctr[st]), words * 4) != cudaSuccess)
        return bail(fail(CS_ERR_OOM, "cudaMalloc of the Stream-K workspace failed"));
      if (cudaMemset(p->split_ctr[st], 0, words * 4) != cudaSuccess) return bail(fail(CS_ERR_CUDA, "cudaMemset failed"));
    }
    size_t pf = 0;
    if (attn && st == 1 && g.kv > 0) {
      // attention pieces: [query block][head][piece][ATT_PART_COLS][128 rows]
      pf = static_cast<size_t>(g.m_blocks) * g.n_tiles[st] * g.kv_max * cs::ATT_PART_COLS * cs::BM;
    } else if (g.splits[st] > 1) {
      const int acc_n = (desc->kind == CS_CHAIN_MLP_SWIGLU && st == 0) ? 256 : g.bn[st];
      pf = static_cast<size_t>(g.splits[st]) * g.m_blocks * g.n_tiles[st] * cs::BM * acc_n;
    }
    if (pf == 0) continue;
    p->partial_bytes[st] = pf * 4;
    const size_t words = static_cast<size_t>(g.m_blocks) * g.n_tiles[st];
    if (cudaMalloc(reinterpret_cast<void**>(&p->partial[st]), pf * 4) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&p->split_ctr[st]), words * 4) != cudaSuccess)
      return bail(fail(CS_ERR_OOM, "cudaMalloc of the split-K workspace failed"));
    if (cudaMemset(p->split_ctr[st], 0, words * 4) != cudaSuccess) return bail(fail(CS_ERR_CUDA, "cudaMemset failed"));
  }
  if (cudaMemset(p->ctrl, 0, cs::CTRL_WORDS * 4) != cudaSuccess) return bail(fail(CS_ERR_CUDA, "cudaMemset failed"));
  const Sched fused = build_fused(g);
  p->n_fused = fused.n_units;
  if ((s = upload(&p->sched_fused, fused.v)) != CS_OK) return bail(s);
  for (int st = 0; st < g.stages; ++st) {
    const Sched one = build_stage(g, st);
    p->n_stage[st] = one.n_units;
    if ((s = upload(&p->sched_stage[st], one.v)) != CS_OK) return bail(s);
  }
  // plan-owned intermediate maps (never re-encoded)
  int owned[5];
  int n_owned = 0;
  if (attn) {
    if ((s = encode_act(p, AMAP_QKVST, p->inter[0], desc->M, 3 * desc->F, true)) != CS_OK) return bail(s);
    if ((s = encode_act(p, AMAP_QKVLD, p->inter[0], desc->M, 3 * desc->F, false)) != CS_OK) return bail(s);
    if ((s = encode_act(p, AMAP_OST, p->inter[1], desc->M, desc->F, true)) != CS_OK) return bail(s);
    if ((s = encode_act(p, AMAP_OLD, p->inter[1], desc->M, desc->F, false)) != CS_OK) return bail(s);
    if ((s = encode_2d(&p->maps[AMAP_K64], p->inter[0], desc->dtype == CS_BF16, 3 * desc->F, desc->M, 64, 64)) !=
        CS_OK)
      return bail(s);
    owned[0] = AMAP_QKVST, owned[1] = AMAP_QKVLD, owned[2] = AMAP_OST, owned[3] = AMAP_OLD, owned[4] = AMAP_K64;
    n_owned = 5;
  } else {
    if ((s = encode_act(p, MAP_HST, p->inter[0], desc->M, desc->F, true)) != CS_OK) return bail(s);
    if ((s = encode_act(p, MAP_HLD, p->inter[0], desc->M, desc->F, false, a_rows(p))) != CS_OK)
      return bail(s);
    owned[0] = MAP_HST, owned[1] = MAP_HLD;
    n_owned = 2;
  }
  bool is_owned[kMaxMaps] = {};
  for (int i = 0; i < n_owned; ++i) {
    is_owned[owned[i]] = true;
    p->slots[owned[i]].ptr = nullptr;
  }
  // unused map slots must still hold a well-formed descriptor for the prefetch
  for (int i = 0; i < kMaxMaps; ++i)
    if (!is_owned[i]) {
      std::memcpy(&p->maps[i], &p->maps[owned[0]], sizeof(CUtensorMap));
      p->slots[i].valid = false;
    }
  *out = p;
  return CS_OK;
}

cs_status cs_chain_destroy(cs_chain_t p) {
  if (!p) return CS_OK;
  cudaSetDevice(p->device);
  cudaDeviceSynchronize();
  free_plan(p);
  return CS_OK;
}

cs_status cs_mlp_forward(cs_chain_t p, const cs_mlp_args* a, void* stream) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  if (p->d.kind == CS_CHAIN_ATTN) return fail(CS_ERR_INVALID_ARG, "plan is an attention chain");
  if (p->error_latched) return fail(CS_ERR_NEEDS_RESET, "plan holds a device error; call cs_chain_reset");
  cs_status s = bind_mlp(p, a);
  if (s != CS_OK) return s;
  cs::KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  fill_common(p, kp);
  fill_mlp_stages(p, a, kp);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p->d.policy == CS_SYNC_STREAM) {
    kp.waits = 0;
    kp.release = 1;
    kp.bump_epoch = 0;
    if ((s = launch(p, kp, p->sched_stage[0], p->n_stage[0], st)) != CS_OK) return s;
    kp.bump_epoch = 1;
    next_trace_segment(p, kp, 0);
    return launch(p, kp, p->sched_stage[1], p->n_stage[1], st);
  }
  kp.waits = 1;
  kp.release = 1;
  kp.bump_epoch = 1;
  return launch(p, kp, p->sched_fused, p->n_fused, st);
}

cs_status cs_mlp_forward_host(cs_chain_t p, const cs_mlp_args* a, void* stream) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  if (!a || !a->X || !a->Y) return fail(CS_ERR_INVALID_ARG, "host X and Y are required");
  if (p->d.kind == CS_CHAIN_ATTN) return fail(CS_ERR_INVALID_ARG, "plan is an attention chain");
  const size_t bytes = static_cast<size_t>(p->d.M) * p->d.H * 2;
  CS_CUDA(cudaSetDevice(p->device));
  if (!p->s_h2d) {
    for (int b = 0; b < 2; ++b)
      if (cudaMalloc(&p->host_x[b], bytes) != cudaSuccess || cudaMalloc(&p->host_y[b], bytes) != cudaSuccess)
        return fail(CS_ERR_OOM, "cudaMalloc of the host-path buffers failed");
    for (cudaEvent_t* evs : {p->ev_x, p->ev_k, p->ev_y})
      for (int i = 0; i < 2; ++i)
        if (cudaEventCreateWithFlags(&evs[i], cudaEventDisableTiming) != cudaSuccess)
          return fail(CS_ERR_CUDA, "cudaEventCreate failed");
    if (cudaStreamCreateWithFlags(&p->s_h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p->s_d2h, cudaStreamNonBlocking) != cudaSuccess)
      return fail(CS_ERR_CUDA, "cudaStreamCreate failed");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int b = static_cast<int>(p->host_calls & 1u);
  // X[b] was last read by the forward of call i-2; Y[b] last copied out by its read-back
  // (waits on events not yet recorded complete at once)
  CS_CUDA(cudaStreamWaitEvent(p->s_h2d, p->ev_k[b], 0));
  CS_CUDA(cudaMemcpyAsync(p->host_x[b], a->X, bytes, cudaMemcpyHostToDevice, p->s_h2d));
  CS_CUDA(cudaEventRecord(p->ev_x[b], p->s_h2d));
  CS_CUDA(cudaStreamWaitEvent(st, p->ev_x[b], 0));
  CS_CUDA(cudaStreamWaitEvent(st, p->ev_y[b], 0));
  cs_mlp_args dev = *a;
  dev.X = p->host_x[b];
  dev.Y = p->host_y[b];
  cs_status s = cs_mlp_forward(p, &dev, stream);
  if (s != CS_OK) return s;
  CS_CUDA(cudaEventRecord(p->ev_k[b], st));
  CS_CUDA(cudaStreamWaitEvent(p->s_d2h, p->ev_k[b], 0));
  CS_CUDA(cudaMemcpyAsync(a->Y, p->host_y[b], bytes, cudaMemcpyDeviceToHost, p->s_d2h));
  CS_CUDA(cudaEventRecord(p->ev_y[b], p->s_d2h));
  ++p->host_calls;
  return CS_OK;
}

cs_status cs_chain_host_join(cs_chain_t p, void* stream) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  if (!p->s_h2d) return CS_OK;
  for (int b = 0; b < 2; ++b) CS_CUDA(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), p->ev_y[b], 0));
  return CS_OK;
}

cs_status cs_attn_chain_forward(cs_chain_t p, const cs_attn_args* a, void* stream) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  if (p->d.kind != CS_CHAIN_ATTN) return fail(CS_ERR_INVALID_ARG, "plan is not an attention chain");
  if (p->error_latched) return fail(CS_ERR_NEEDS_RESET, "plan holds a device error; call cs_chain_reset");
  cs_status s = bind_attn(p, a);
  if (s != CS_OK) return s;
  cs::KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  fill_common(p, kp);
  fill_attn_stages(p, kp);
  fill_attn_prefetch(p, a, kp);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p->d.policy == CS_SYNC_STREAM) {
    kp.waits = 0;
    kp.release = 1;
    for (int stg = 0; stg < 3; ++stg) {
      kp.bump_epoch = stg == 2;
      if (stg > 0) next_trace_segment(p, kp, stg - 1);
      if ((s = launch(p, kp, p->sched_stage[stg], p->n_stage[stg], st)) != CS_OK) return s;
    }
    return CS_OK;
  }
  kp.waits = 1;
  kp.release = 1;
  kp.bump_epoch = 1;
  return launch(p, kp, p->sched_fused, p->n_fused, st);
}

cs_status cs_chain_forward_stage(cs_chain_t p, const void* args, int stage, void* stream) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  if (p->error_latched) return fail(CS_ERR_NEEDS_RESET, "plan holds a device error; call cs_chain_reset");
  if (stage < 0 || stage >= p->stages) return fail(CS_ERR_INVALID_ARG, "stage %d out of range", stage);
  cs::KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  cs_status s;
  if (p->d.kind == CS_CHAIN_ATTN) {
    const cs_attn_args* a = static_cast<const cs_attn_args*>(args);
    if ((s = bind_attn(p, a)) != CS_OK) return s;
    fill_common(p, kp);
    fill_attn_stages(p, kp);
    fill_attn_prefetch(p, a, kp);
  } else {
    const cs_mlp_args* a = static_cast<const cs_mlp_args*>(args);
    if ((s = bind_mlp(p, a)) != CS_OK) return s;
    fill_common(p, kp);
    fill_mlp_stages(p, a, kp);
  }
  kp.waits = 0;
  kp.release = 0;
  kp.bump_epoch = 0;
  return launch(p, kp, p->sched_stage[stage], p->n_stage[stage], static_cast<cudaStream_t>(stream));
}

cs_status cs_chain_status(cs_chain_t p) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  uint32_t w[cs::CTRL_WORDS];
  CS_CUDA(cudaMemcpy(w, p->ctrl, sizeof(w), cudaMemcpyDeviceToHost));
  if (w[cs::CTRL_ERROR] == 0) return CS_OK;
  p->error_latched = true;
  const cs_status code = static_cast<cs_status>(w[cs::CTRL_ERROR]);
  return fail(code, "device error %u: unit 0x%08x where 0x%x cta %u", w[cs::CTRL_ERROR], w[cs::CTRL_ERR_UNIT],
              w[cs::CTRL_ERR_WHERE], w[cs::CTRL_ERR_CTA]);
}

cs_status cs_chain_reset(cs_chain_t p) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  CS_CUDA(cudaDeviceSynchronize());
  for (int b = 0; b < 3; ++b)
    if (p->sems[b]) CS_CUDA(cudaMemset(p->sems[b], 0, (p->sem_words[b] + p->m_tiles) * 4));
  CS_CUDA(cudaMemset(p->ctrl, 0, cs::CTRL_WORDS * 4));
  for (int st = 0; st < p->stages; ++st)
    if (p->split_ctr[st])
      CS_CUDA(cudaMemset(p->split_ctr[st], 0, static_cast<size_t>(p->m_blocks) * p->n_tiles[st] * 4));
  CS_CUDA(cudaDeviceSynchronize());
  p->error_latched = false;
  return CS_OK;
}

cs_status cs_chain_query(cs_chain_t p, cs_chain_info* info) {
  if (!p || !info) return fail(CS_ERR_INVALID_ARG, "NULL argument");
  info_geometry(p, p->n_fused, info);
  info->intermediate[0] = p->inter[0];
  info->intermediate[1] = p->inter[1];
  info->sem_words[0] = p->sem_words[0];
  info->sem_words[1] = p->sem_words[1];
  const int last = p->stages - 1;
  info->out_tile_sems = p->sems[last];
  info->out_row_sems = p->sems[last] ? p->sems[last] + p->sem_words[last] : nullptr;
  info->out_sem_words = p->sems[last] ? p->sem_words[last] : 0;
  return CS_OK;
}

cs_status cs_tune_match(const cs_chain_desc* desc, int num_sms, int* entry, cs_chain_desc* resolved) {
  if (!entry) return fail(CS_ERR_INVALID_ARG, "entry is NULL");
  *entry = -1;
  cs_status s = validate(desc);
  if (s != CS_OK) return s;
  if (num_sms < 1) return fail(CS_ERR_INVALID_ARG, "num_sms=%d", num_sms);
  const cs_chain_desc rd = resolve_desc(desc, num_sms, entry);
  if (resolved) *resolved = rd;
  return CS_OK;
}

cs_status cs_chain_plan_info(const cs_chain_desc* desc, int num_sms, cs_chain_info* info) {
  if (!info) return fail(CS_ERR_INVALID_ARG, "info is NULL");
  cs_status s = validate(desc);
  if (s != CS_OK) return s;
  if (num_sms < 1) return fail(CS_ERR_INVALID_ARG, "num_sms=%d", num_sms);
  cs_chain_s p;
  p.num_sms = desc->num_sms > 0 && desc->num_sms < num_sms ? desc->num_sms : num_sms;
  p.d = resolve_desc(desc, p.num_sms, &p.tuned_entry);
  const Geometry g = geometry(&p.d, p.num_sms);
  shape_plan(&p, g, desc->kind, desc->M);
  info_geometry(&p, build_fused(g).n_units, info);
  return CS_OK;
}

int cs_library_features(void) { return kClusterMulticast ? CS_FEATURE_CLUSTER_MULTICAST : 0; }

cs_status cs_chain_debug_read_sems(cs_chain_t p, int boundary, uint32_t* host, size_t n, uint32_t* epoch) {
  if (!p || !host) return fail(CS_ERR_INVALID_ARG, "NULL argument");
  if (boundary < 0 || boundary >= p->stages || !p->sems[boundary])
    return fail(CS_ERR_INVALID_ARG, "boundary %d has no semaphores", boundary);
  const size_t words = p->sem_words[boundary] + p->m_tiles;
  if (n < words) return fail(CS_ERR_INVALID_ARG, "need %zu words, got %zu", words, n);
  CS_CUDA(cudaMemcpy(host, p->sems[boundary], words * 4, cudaMemcpyDeviceToHost));
  if (epoch) CS_CUDA(cudaMemcpy(epoch, p->ctrl + cs::CTRL_EPOCH, 4, cudaMemcpyDeviceToHost));
  return CS_OK;
}

cs_status cs_chain_debug_set_delays(cs_chain_t p, int stage, const uint32_t* ns, size_t n) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  if (stage < 0 || stage >= p->stages - 1) return fail(CS_ERR_INVALID_ARG, "stage %d has no consumers", stage);
  if (!ns || n == 0) {
    if (p->delays[stage]) cudaFree(p->delays[stage]);
    p->delays[stage] = nullptr;
    return CS_OK;
  }
  if (n != static_cast<size_t>(p->units[stage])) return fail(CS_ERR_INVALID_ARG, "need %d delays", p->units[stage]);
  if (!p->delays[stage] && cudaMalloc(reinterpret_cast<void**>(&p->delays[stage]), n * 4) != cudaSuccess)
    return fail(CS_ERR_OOM, "cudaMalloc failed");
  CS_CUDA(cudaMemcpy(p->delays[stage], ns, n * 4, cudaMemcpyHostToDevice));
  return CS_OK;
}

cs_status cs_chain_debug_skip_release(cs_chain_t p, int stage, int unit) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  if (stage < 0 || stage >= p->stages - 1) return fail(CS_ERR_INVALID_ARG, "stage %d has no consumers", stage);
  if (unit < -1 || unit >= p->units[stage]) return fail(CS_ERR_INVALID_ARG, "unit %d out of range", unit);
  p->skip[stage] = unit;
  return CS_OK;
}

cs_status cs_chain_debug_copy_intermediate(cs_chain_t p, int which, void* dst, size_t bytes) {
  if (!p || !dst) return fail(CS_ERR_INVALID_ARG, "NULL argument");
  if (which < 0 || which > 1 || !p->inter[which]) return fail(CS_ERR_INVALID_ARG, "no intermediate %d", which);
  if (bytes > p->inter_bytes[which]) return fail(CS_ERR_INVALID_ARG, "%zu bytes > buffer (%zu)", bytes, p->inter_bytes[which]);
  CS_CUDA(cudaDeviceSynchronize());
  CS_CUDA(cudaMemcpy(dst, p->inter[which], bytes, cudaMemcpyDeviceToDevice));
  return CS_OK;
}

cs_status cs_chain_debug_poison_intermediate(cs_chain_t p, int which, void* stream) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  if (which < -1 || which > 2) return fail(CS_ERR_INVALID_ARG, "which=%d (-1..2)", which);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // all-ones bytes: NaN as fp16, bf16 and fp32
  for (int b = 0; b < 2; ++b)
    if ((which == -1 || which == b) && p->inter[b]) CS_CUDA(cudaMemsetAsync(p->inter[b], 0xFF, p->inter_bytes[b], st));
  if ((which == -1 || which == 2) && p->sk_partial) {
    const size_t bytes = static_cast<size_t>(p->sk_tiles) * p->sk_max_nc * p->cl * cs::BM * p->bn[p->stages - 1] * 4;
    CS_CUDA(cudaMemsetAsync(p->sk_partial, 0xFF, bytes, st));
  }
  if (which == -1 || which == 2)
    for (int stg = 0; stg < p->stages; ++stg)
      if (p->partial[stg]) CS_CUDA(cudaMemsetAsync(p->partial[stg], 0xFF, p->partial_bytes[stg], st));
  return CS_OK;
}

cs_status cs_chain_debug_set_epoch(cs_chain_t p, uint32_t epoch) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  CS_CUDA(cudaDeviceSynchronize());
  // every counter as it stands after `epoch` complete forwards, modulo 2^32
  for (int b = 0; b < 3; ++b) {
    if (!p->sems[b]) continue;
    std::vector<uint32_t> v(p->sem_words[b] + p->m_tiles, epoch);
    for (int m = 0; m < p->m_tiles; ++m) v[p->sem_words[b] + m] = epoch * static_cast<uint32_t>(p->n_tiles[b]);
    CS_CUDA(cudaMemcpy(p->sems[b], v.data(), v.size() * 4, cudaMemcpyHostToDevice));
  }
  for (int stg = 0; stg < p->stages; ++stg)
    if (p->split_ctr[stg]) {
      std::vector<uint32_t> v(static_cast<size_t>(p->m_blocks) * p->n_tiles[stg],
                              epoch * static_cast<uint32_t>(p->splits[stg]));
      if (p->d.kind == CS_CHAIN_ATTN && stg == 1 && p->kv > 0) {
        // one arrival per piece of the query block's tile row
        for (int qb = 0; qb < p->m_blocks; ++qb)
          for (int h = 0; h < p->n_tiles[stg]; ++h)
            v[static_cast<size_t>(qb) * p->n_tiles[stg] + h] = epoch * static_cast<uint32_t>((qb / p->cg + p->kv) / p->kv);
      }
      if (stg == p->stages - 1 && p->sk_units > 0) {
        // a Stream-K tile counts one arrival per contributing unit (per 128-row block)
        std::vector<uint32_t> table(static_cast<size_t>(p->sk_tiles));
        CS_CUDA(cudaMemcpy(table.data(), p->sched_fused + p->n_fused, table.size() * 4, cudaMemcpyDeviceToHost));
        const long long K = p->k_iters[stg], q = p->sk_q;
        for (int j = 0; j < p->sk_tiles; ++j) {
          const uint32_t nc = static_cast<uint32_t>(((j + 1) * K - 1) / q - (j * K) / q + 1);
          const int m = static_cast<int>((table[j] >> 14) & 0xFFFu), n = static_cast<int>(table[j] & 0x3FFFu);
          for (int r = 0; r < p->cl; ++r) v[static_cast<size_t>(m * p->cl + r) * p->n_tiles[stg] + n] = epoch * nc;
        }
      }
      CS_CUDA(cudaMemcpy(p->split_ctr[stg], v.data(), v.size() * 4, cudaMemcpyHostToDevice));
    }
  CS_CUDA(cudaMemcpy(p->ctrl + cs::CTRL_EPOCH, &epoch, 4, cudaMemcpyHostToDevice));
  CS_CUDA(cudaDeviceSynchronize());
  return CS_OK;
}

cs_status cs_chain_debug_trace(cs_chain_t p, int enable) {
  if (!p) return fail(CS_ERR_INVALID_ARG, "plan is NULL");
  if (p->trace) {
    cudaFree(p->trace);
    p->trace = nullptr;
    p->trace_records = 0;
  }
  if (!enable) return CS_OK;
  int per_stage = 0;
  for (int st = 0; st < p->stages; ++st) per_stage += p->n_stage[st];
  const int recs = std::max(p->n_fused, per_stage) * p->cl;
  const size_t bytes = static_cast<size_t>(recs) * cs::TRACE_WORDS * 8;
  if (cudaMalloc(reinterpret_cast<void**>(&p->trace), bytes) != cudaSuccess) return fail(CS_ERR_OOM, "cudaMalloc failed");
  CS_CUDA(cudaMemset(p->trace, 0, bytes));
  p->trace_records = recs;
  return CS_OK;
}

cs_status cs_chain_debug_read_trace(cs_chain_t p, uint64_t* host, size_t n, size_t* n_out) {
  if (!p || !n_out) return fail(CS_ERR_INVALID_ARG, "NULL argument");
  *n_out = static_cast<size_t>(p->trace_records);
  if (!p->trace || n == 0) return CS_OK;
  if (!host) return fail(CS_ERR_INVALID_ARG, "host is NULL");
  const size_t m = n < *n_out ? n : *n_out;
  CS_CUDA(cudaMemcpy(host, p->trace, m * cs::TRACE_WORDS * 8, cudaMemcpyDeviceToHost));
  return CS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free forward
// Scratch of cs_mlp_forward_noalloc: one array per device that loads the
// library.  In host code `g_noalloc_scratch` names a host-side stand-in, not
// device memory, so its device address is looked up per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CS_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_ptr[kMaxDevices] = {};

// Device address of this device's scratch array (looked up once per device,
// with that device current).
cs_status noalloc_scratch(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(CS_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return fail(CS_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = static_cast<unsigned char*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return CS_OK;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Per call, in stream order before the chain: zero the control block and the
// semaphores, and write the fused and per-stage schedules from the closed form,
// one thread per word (nothing is copied from host memory).
__global__ void noalloc_prep_kernel(cs::SchedGeo g, uint32_t* zero, long long n_zero, uint32_t* fused,
                                    long long n_fused, uint32_t* st0, long long n0, uint32_t* st1, long long n1) {
  const long long total = n_zero + n_fused + n0 + n1;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    long long j = i;
    if (j < n_zero) {
      zero[j] = 0u;
      continue;
    }
    j -= n_zero;
    if (j < n_fused) {
      fused[j] = cs::sched_fused_entry(g, j);
      continue;
    }
    j -= n_fused;
    if (j < n0) {
      st0[j] = cs::sched_stage_entry(g, 0, j);
      continue;
    }
    j -= n0;
    st1[j] = cs::sched_stage_entry(g, 1, j);
  }
}

}  // namespace

extern "C" {

cs_status cs_mlp_forward_noalloc(const cs_chain_desc* desc, const cs_mlp_args* args, void* stream) {
  cs_status s = validate(desc);
  if (s != CS_OK) return s;
  if (desc->kind == CS_CHAIN_ATTN) return fail(CS_ERR_UNSUPPORTED, "the allocation-free forward runs MLP chains only");
  if (desc->out_release) return fail(CS_ERR_UNSUPPORTED, "the allocation-free forward has no output semaphores");
  if (desc->split_k > 1)
    return fail(CS_ERR_UNSUPPORTED, "split_k=%d: the allocation-free forward runs unsplit tiles (split_k 0 or 1)",
                desc->split_k);
  if (desc->split_k_first > 1)
    return fail(CS_ERR_UNSUPPORTED,
                "split_k_first=%d: the allocation-free forward runs unsplit tiles (split_k_first 0 or 1)",
                desc->split_k_first);
  if (desc->sk_tiles > 0)
    return fail(CS_ERR_UNSUPPORTED, "sk_tiles=%d: the allocation-free forward has no Stream-K workspace",
                desc->sk_tiles);
  int sms = 0;
  const int dev = device_sms(&sms);
  if (dev < 0) return fail(CS_ERR_CUDA, "no CUDA device available");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major * 10 + minor != 103)
    return fail(CS_ERR_UNSUPPORTED, "device is sm_%d%d; this library is built for sm_103a only", major, minor);

  // A plan on the host stack whose buffers all point into the scratch array.
  // The tuning table is not consulted; policy AUTO runs TILE.
  cs_chain_s p;
  p.d = *desc;
  p.d.split_k = 1;  // no split-K workspace in the fixed array
  p.d.split_k_first = 0;
  p.d.sk_tiles = -1;
  if (p.d.policy == CS_SYNC_AUTO) p.d.policy = CS_SYNC_TILE;
  p.device = dev;
  p.num_sms = desc->num_sms > 0 && desc->num_sms < sms ? desc->num_sms : sms;
  Geometry g = geometry(&p.d, p.num_sms);
  shape_plan(&p, g, desc->kind, desc->M);
  if ((s = resident_workers(&p, &p.workers)) != CS_OK) return s;
  const cs::SchedGeo sg = sched_geo(g);
  const long long n_fused = cs::sched_fused_count(sg);
  const long long n_st0 = cs::sched_stage_count(sg, 0), n_st1 = cs::sched_stage_count(sg, 1);
  p.n_fused = static_cast<int>(n_fused);

  // Carve the array: control block and semaphores (cleared every call), then
  // the schedules, then the intermediate H [M, F].
  p.sem_words[0] = static_cast<size_t>(g.m_blocks) * g.n_tiles[0];
  const size_t zero_words = cs::CTRL_WORDS + p.sem_words[0] + g.m_blocks;
  const size_t sched_words = static_cast<size_t>(n_fused + n_st0 + n_st1);
  const size_t h_off = align256((zero_words + sched_words) * 4);
  p.inter_bytes[0] = static_cast<size_t>(desc->M) * desc->F * 2;
  const size_t need = h_off + p.inter_bytes[0];
  if (need > CS_NOALLOC_SCRATCH_BYTES)
    return fail(CS_ERR_INVALID_ARG,
                "M=%d F=%d needs %zu bytes of scratch; the allocation-free forward has %u (use cs_chain_plan)",
                desc->M, desc->F, need, CS_NOALLOC_SCRATCH_BYTES);
  unsigned char* base = nullptr;
  if ((s = noalloc_scratch(dev, &base)) != CS_OK) return s;
  uint32_t* words = reinterpret_cast<uint32_t*>(base);
  p.ctrl = words;
  p.sems[0] = words + cs::CTRL_WORDS;
  p.sched_fused = words + zero_words;
  p.sched_stage[0] = p.sched_fused + n_fused;
  p.sched_stage[1] = p.sched_stage[0] + n_st0;
  p.inter[0] = base + h_off;

  // Tensor maps of the intermediate (in the array) and of the caller's tensors.
  if ((s = encode_act(&p, MAP_HST, p.inter[0], desc->M, desc->F, true)) != CS_OK) return s;
  if ((s = encode_act(&p, MAP_HLD, p.inter[0], desc->M, desc->F, false, a_rows(&p))) != CS_OK) return s;
  for (int i = 0; i < kMaxMaps; ++i)
    if (i != MAP_HST && i != MAP_HLD) std::memcpy(&p.maps[i], &p.maps[MAP_HLD], sizeof(CUtensorMap));
  if ((s = bind_mlp(&p, args)) != CS_OK) return s;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  {
    const long long total = static_cast<long long>(zero_words) + n_fused + n_st0 + n_st1;
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<long long>((total + threads - 1) / threads, 4 * sms));
    noalloc_prep_kernel<<<blocks, threads, 0, st>>>(sg, words, static_cast<long long>(zero_words), p.sched_fused,
                                                     n_fused, p.sched_stage[0], n_st0, p.sched_stage[1], n_st1);
    CS_CUDA(cudaGetLastError());
  }

  cs::KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  fill_common(&p, kp);
  fill_mlp_stages(&p, args, kp);
  kp.release = 1;
  if (desc->policy == CS_SYNC_STREAM) {
    kp.waits = 0;
    kp.bump_epoch = 0;
    if ((s = launch(&p, kp, p.sched_stage[0], p.sched_units[0], st)) != CS_OK) return s;
    kp.bump_epoch = 1;
    return launch(&p, kp, p.sched_stage[1], p.sched_units[1], st);
  }
  kp.waits = 1;
  kp.bump_epoch = 1;
  return launch(&p, kp, p.sched_fused, p.n_fused, st);
}

cs_status cs_noalloc_status(void) {
  int dev = 0;
  CS_CUDA(cudaGetDevice(&dev));
  unsigned char* base = nullptr;
  cs_status s = noalloc_scratch(dev, &base);
  if (s != CS_OK) return s;
  uint32_t w[cs::CTRL_WORDS];
  CS_CUDA(cudaMemcpy(w, base, sizeof(w), cudaMemcpyDeviceToHost));
  if (w[cs::CTRL_ERROR] == 0) return CS_OK;
  return fail(static_cast<cs_status>(w[cs::CTRL_ERROR]), "device error %u: unit 0x%08x where 0x%x cta %u",
              w[cs::CTRL_ERROR], w[cs::CTRL_ERR_UNIT], w[cs::CTRL_ERR_WHERE], w[cs::CTRL_ERR_CTA]);
}

}  // extern "C"
