/*
 * cs_chain.h -- C ABI of a tile-synchronised GEMM-chain library for GB300 (sm_103a).
 *
 * What it computes.  A chain of dependent GEMMs on one GPU, for example a
 * transformer MLP  Y = GeLU(X W1 + b1) W2  (CuSync README, MLP paragraph:
 * "8 way model parallelism GPT3 175B (H=12288 FP16) and LLAMA 65.2B
 * (H=8192)", with GeLU fused into the first GEMM).  The consumer GEMM's
 * thread-block tiles start as soon as the producer tiles they read are
 * finished, instead of at the kernel boundary (CuSync README, first
 * paragraph: a programmer writes policies that synchronise dependent tiles
 * of a producer/consumer kernel chain, which raises utilisation in the last
 * thread-block wave).  The result is the plain composed chain; only the
 * timing changes.
 *
 * How.  One persistent kernel per forward call: a dependency-ordered tile
 * scheduler hands producer and consumer tile units to the SMs; tcgen05 MMAs
 * accumulate in tensor memory, fed by TMA into a multi-stage shared-memory
 * ring; the producer epilogue (bias + activation, downcast, TMA store) then
 * release-increments a per-tile semaphore in global memory; the consumer's
 * TMA warp acquire-waits on those semaphores per K-slice before loading the
 * intermediate.  The wait policy is selectable (cs_policy).
 *
 * Conventions for every entry point.
 *  - Every entry point returns a cs_status and never aborts the process.
 *    On failure, cs_last_error_string() (thread-local) says why.
 *  - Matrices are row-major, contiguous, with 16-byte aligned base pointers.
 *    Device pointers are CUDA device (or managed) memory on the device that
 *    was current when the plan was made; the caller owns them.
 *  - "stream" is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Forward calls only enqueue work; device-side failures surface
 *    through cs_chain_status() after the caller synchronises the stream.
 *  - A plan is not thread-safe and must be used by one stream at a time: its
 *    semaphores and intermediate buffers are per plan.
 */
#ifndef CS_CHAIN_H
#define CS_CHAIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CS_ABI_VERSION 7

typedef struct cs_chain_s* cs_chain_t;

typedef enum cs_status {
  CS_OK = 0,
  CS_ERR_INVALID_ARG = 1,  /* NULL/misaligned pointer, bad shape or enum value */
  CS_ERR_UNSUPPORTED = 2,  /* well-formed request this build does not implement */
  CS_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed (see cs_last_error_string) */
  CS_ERR_TIMEOUT = 4,      /* a consumer tile gave up waiting for a producer tile */
  CS_ERR_OOM = 5,          /* device allocation failed */
  CS_ERR_WATCHDOG = 6,     /* an in-CTA pipeline wait exceeded its limit (internal error) */
  CS_ERR_NEEDS_RESET = 7   /* the plan holds a device error; call cs_chain_reset() */
} cs_status;

typedef enum cs_dtype { CS_F16 = 0, CS_BF16 = 1 } cs_dtype;

/* Which chain the plan runs.
 *  MLP_GELU : H = GeLU_tanh(X W1 + b1),  Y = H W2            (GPT-3 MLP shard)
 *  MLP_SWIGLU: H = SiLU(X Wg) * (X Wu),  Y = H Wd            (LLaMA MLP shard)
 *  ATTN     : QKV = X Wqkv; O = per-head causal softmax(Q K^T/sqrt(d)) V;
 *             Y = O Wo                                         (attention shard)
 * GeLU_tanh(x) = x/2 (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))), SiLU(x) = x/(1+e^-x). */
typedef enum cs_chain_kind { CS_CHAIN_MLP_GELU = 0, CS_CHAIN_MLP_SWIGLU = 1, CS_CHAIN_ATTN = 2 } cs_chain_kind;

/* When a consumer tile may read the intermediate (CuSync README, first paragraph:
 * policies over dependent tiles).  A producer tile covers 128 rows x tile_n columns
 * of the intermediate; a consumer K-slice of 64 columns lies inside one of them.
 *  TILE    : wait for the one producer tile that wrote the K-slice.
 *  ROW     : wait for every producer tile of the consumer's 128-row block.
 *  STRIDED : wait for every producer tile of the row block whose column-tile index
 *            is congruent (mod stride) to the one that wrote the K-slice.  With
 *            stride = heads this is "the Q, K and V tiles of one head".
 *  STREAM  : two-kernel control: all producer tiles in one launch, all consumer
 *            tiles in a second launch on the same stream, no tile waits.
 *  AUTO    : (desc only) the fastest fused policy (TILE, ROW or STRIDED) that the
 *            loaded tuning table recorded for this chain shape at the nearest
 *            measured M; TILE when the table has no entry.  All policies give the
 *            same bits; only the timing differs.                               */
typedef enum cs_policy {
  CS_SYNC_AUTO = -1,
  CS_SYNC_TILE = 0,
  CS_SYNC_ROW = 1,
  CS_SYNC_STRIDED = 2,
  CS_SYNC_STREAM = 3
} cs_policy;

/* Storage layout of every weight matrix of the chain.
 *  KN : W stored as in the maths, [K, N] row-major (W1 is [H, F]).
 *  NK : W stored transposed, [N, K] row-major (W1 is [F, H]; torch.nn.Linear). */
typedef enum cs_weight_layout { CS_WEIGHTS_KN = 0, CS_WEIGHTS_NK = 1 } cs_weight_layout;

typedef struct cs_chain_desc {
  int kind;            /* cs_chain_kind */
  int M;               /* rows (tokens; for ATTN also the causal sequence length),
                          1 .. 524160 */
  int H;               /* model width: GEMM1 K and GEMM2 N; multiple of 8 */
  int F;               /* MLP: FFN shard width (GEMM1 N, GEMM2 K), multiple of 8.
                          ATTN: heads * head_dim.                                   */
  int dtype;           /* cs_dtype of X, weights, bias, intermediate and Y; fp32 accumulate */
  int policy;          /* cs_policy */
  int weight_layout;   /* cs_weight_layout */
  int stride;          /* CS_SYNC_STRIDED stride in producer column tiles; 0 = auto
                          (heads for ATTN, 4 for MLPs)                               */
  int heads;           /* ATTN only: number of heads */
  int head_dim;        /* ATTN only: must be 128 */
  int num_sms;         /* persistent grid size; 0 = every SM of the device */
  int lag;             /* schedule: producer row-block groups issued before the
                          first consumer group; -1 = auto (1)                       */
  int group_m;         /* schedule: tile rows per rasterisation group (units of a
                          group run column-tile-major so concurrent tiles share
                          weights in L2); 0 = auto (at most 1024 rows per group;
                          with 256-row pair tiles at least two groups; GeLU chains
                          on 512-row tiles from three tile rows: up to 2048 rows)   */
  int tile_n;          /* output columns per GEMM tile: 64, 128 or 256; 0 = auto
                          (never 64).  SwiGLU producer tiles are always 128
                          (gate|up = 256).  64 runs on single SMs only (tile_m
                          128, MLP chains): twice the tiles of 128 for a stage
                          with fewer tiles than SMs, without K-splits.            */
  int tile_m;          /* rows per GEMM tile: 128 (one SM), 256 (a 2-SM cluster
                          sharing one tcgen05 MMA) or 512 (two such pairs in a 4-CTA
                          cluster that fetch every weight box once and multicast it
                          to both pairs).  256 and 512 run 256-wide tiles: tile_n =
                          128 is refused, and with tile_n = 0 they fall back to 128
                          rows where the automatic tile_n is 128.  SwiGLU pairs hold
                          the gate rows of B on one CTA and the up rows on the other.
                          0 = auto: MLPs take 512 from four 128-row blocks (M > 384;
                          GeLU only where it adds no padding rows over 256), else
                          256 (with 256-wide tiles) for exactly two
                          128-row blocks or from eight, else 128.
                          The attention chain runs 128 (with tile_n 128) or 256 (with
                          tile_n 256: attention units of two query blocks on a CTA
                          pair); auto 256 from four 128-row blocks.  Semaphores stay
                          per 128-row block.                                        */
  int split_k;         /* K-splits per GEMM tile: 0 = auto (split when a stage has
                          fewer tiles than the grid, small M), 1 = never, 2..15 = that
                          many for every GEMM stage.  Splits write fp32 partial tiles
                          to a plan-owned workspace; the last split to finish sums
                          them in split order (bit-reproducible) and runs the
                          epilogue and the release.                                  */
  int prefetch;        /* L2 prefetch distance in K-slices: the scheduler warp brings
                          the weight lines (and producer A rows) that far ahead of
                          the TMA loads into L2; 0 = auto (off: measured slower on
                          GB300), -1 = off                                          */
  int raster;          /* order of a stage's tiles inside a row group: 0 = auto
                          (column-major, or the tuning table's choice), 1 =
                          column-major (tiles sharing a weight tile run together,
                          a tile's K-splits one after another), 2 = row-major (row
                          blocks complete one after another, so their consumers
                          can start sooner), 3 = column-major for the first stage
                          and K-range-major for a split later stage: K-split 0 of
                          every tile of the group, then K-split 1, ... A split
                          consumer's K range needs only the producer tiles of that
                          range, so when the producers run in more than one wave
                          (they finish in column-tile order) the first consumers
                          start while the later producer tiles still stream their
                          weights.                                                 */
  int pdl;             /* programmatic dependent launch: a forward queued behind another
                          kernel on the stream starts its CTAs as the earlier grid's
                          CTAs exit, and sets up its barriers and tensor memory while
                          the earlier grid drains; it reads global memory only after
                          that grid has completed (griddepcontrol.wait).  0 = auto
                          (on), 1 = on, -1 = off (plain stream order)               */
  int tuned;           /* 0 = consult the loaded tuning table (cs_tune_load): when
                          tile_m, tile_n, split_k, split_k_first and group_m are
                          all auto, they are taken from the entry of the nearest
                          measured M for this chain shape, dtype, layout and grid
                          size (and raster, where the desc leaves it on auto), and
                          policy AUTO is resolved from it; an entry whose choices
                          do not fit the desc is ignored.  -1 = never (built-in
                          rules only).                                              */
  int out_release;     /* 1: the last stage releases Y the way producers release the
                          intermediate: once a tile of Y is stored, its tile
                          semaphore and its 128-row block's counter are
                          release-incremented (device pointers in cs_chain_info), so
                          that a following consumer of Y -- a collective that sends
                          blocks of rows as they complete, as in the Flux summary's
                          GEMM + reduce-scatter fusion -- may acquire-read a block
                          once its counter reaches epoch * (tiles per row block).
                          Each Y tile then waits for its store to complete before
                          the epilogue moves on.  0 = off.                          */
  unsigned long long spin_timeout_ns; /* per-wait limit of a consumer tile; 0 = 2 s */
  int sk_tiles;        /* Stream-K tail of the last GEMM stage (CuSync README, MLP
                          paragraph: Stream-K as the other fix of the last
                          thread-block wave).  The last sk_tiles tiles of that
                          stage in dispatch order (at most those of the last row
                          group) are not run as tiles; sk_units units instead
                          each take an equal run of their concatenated K-slices,
                          crossing tile boundaries.  A tile's contributing units
                          write fp32 partial tiles to a plan-owned workspace; the
                          last to finish sums them in K order (the same bits on
                          every call and under every policy) and runs the
                          epilogue.  Needs an unsplit last stage: with split_k
                          0 (auto) the last stage then takes no K-splits, with
                          split_k > 1 the tail is not applied.
                          0 = auto (the tuning table's choice, else none),
                          -1 = none, n = that many tiles.                          */
  int sk_units;        /* Stream-K units for those tiles; 0 = one per worker (SM,
                          pair or cluster of the grid).  Each takes at least 8
                          K-slices (fewer units then).                              */
  int kv_chunk;        /* ATTN: key-range pieces of the causal attention units.  A
                          unit of tile row m (tile_m query rows of one head) sees
                          key groups 0..m (tile_m keys each), so the last rows'
                          units are the longest.  With kv_chunk = c the row runs
                          as ceil((m + 1) / c) pieces of at most c key groups, on
                          as many SMs (or pairs) at once; each piece writes its
                          fp32 softmax state (row maximum, row sum, unnormalised
                          output) to a plan-owned workspace, and the last piece of
                          a query block and head to finish merges every piece in
                          piece order (the same bits whichever finishes last),
                          stores O and releases it.  0 = auto (whole rows: the
                          merge costs more than the shorter critical path saves
                          on GB300), -1 = whole rows.  At most 15 pieces per row
                          (c is raised to fit).                                   */
  int split_k_first;   /* K-splits of the first GEMM stage (GEMM1 of an MLP, the
                          QKV GEMM of the attention chain): 0 = as split_k,
                          1..15 = that many (at least 8 K-slices each; with
                          split_k 0 the other stages keep the automatic rule).  A
                          first stage split into more units than the grid runs at
                          once finishes its column tiles in waves, which raster 3
                          lets the consumers use.                                 */
} cs_chain_desc;

/* Fill *desc with defaults (kind MLP_GELU, F16, TILE, KN, auto everything else). */
cs_status cs_chain_desc_init(cs_chain_desc* desc);

/* Make a plan: validates the shapes, builds the tile schedule, allocates the
 * per-tile semaphores, the intermediate buffer(s) and the device control block
 * with cudaMalloc on the current device, and encodes the TMA descriptors of the
 * intermediates.  *out receives the handle (NULL on failure).  The plan fixes M. */
cs_status cs_chain_plan(const cs_chain_desc* desc, cs_chain_t* out);

/* Free everything the plan owns.  NULL-safe.  Synchronises the device first. */
cs_status cs_chain_destroy(cs_chain_t plan);

/* Device pointers of one MLP forward, caller-owned.
 *  X [M,H]; Y [M,H] (written).  MLP_GELU: W1, b1 [F], W2.  MLP_SWIGLU: Wg, Wu, W2 (= Wd).
 *  Weight shapes follow desc.weight_layout: KN -> W1/Wg/Wu [H,F], W2 [F,H];
 *  NK -> W1/Wg/Wu [F,H], W2 [H,F].  Unused pointers may be NULL. */
typedef struct cs_mlp_args {
  const void* X;
  const void* W1;
  const void* b1;
  const void* Wg;
  const void* Wu;
  const void* W2;
  void* Y;
} cs_mlp_args;

/* Enqueue one chain forward on `stream` (one persistent-kernel launch; two for
 * CS_SYNC_STREAM).  TMA descriptors of caller pointers are re-encoded when a
 * pointer changes.  Returns CS_ERR_NEEDS_RESET if an earlier call of this plan
 * reported a device error that has not been cleared. */
cs_status cs_mlp_forward(cs_chain_t plan, const cs_mlp_args* args, void* stream);

/* End-to-end forward from host memory (no counterpart on the pages): args->X
 * (M x H) and args->Y (M x H) are HOST pointers, page-locked for the copies to
 * run asynchronously; weights and bias are device pointers as above.  The plan
 * owns two device buffers for X and two for Y (allocated on the first call)
 * and two copy streams: call i copies X on the first copy stream, runs the
 * forward on `stream` once that copy has landed (and once the read-back of
 * call i-2, which used the same Y buffer, is done), and copies Y back on the
 * second copy stream, so consecutive calls overlap their copies with the
 * kernels.  args->X may be reused or changed as soon as the call's copy has
 * run; args->Y holds the result once cs_chain_host_join has made a stream wait
 * for it and that stream has been synchronised.  The host buffers are the
 * caller's and must stay valid until then. */
cs_status cs_mlp_forward_host(cs_chain_t plan, const cs_mlp_args* args, void* stream);

/* Make `stream` wait until every Y read-back issued by cs_mlp_forward_host on
 * this plan so far has landed in host memory. */
cs_status cs_chain_host_join(cs_chain_t plan, void* stream);

/* Device pointers of one attention-chain forward, caller-owned.
 *  X [M,H]; Wqkv: KN [H, 3F] / NK [3F, H], columns (KN) [Q | K | V], head-major;
 *  Wo: KN [F, H] / NK [H, F]; Y [M,H] (written). */
typedef struct cs_attn_args {
  const void* X;
  const void* Wqkv;
  const void* Wo;
  void* Y;
} cs_attn_args;

/* Enqueue one attention-chain forward (QKV GEMM -> causal attention -> Wo GEMM). */
cs_status cs_attn_chain_forward(cs_chain_t plan, const cs_attn_args* args, void* stream);

/* Run ONE stage of the chain alone, as its own persistent launch with no tile
 * waits and no semaphore releases (the "best standalone GEMM" timing of the
 * effective-overhead measurement; Flux summary, idea I2: total time minus the
 * time of the best unsplit GEMM).  args is a cs_mlp_args* or cs_attn_args* as
 * the plan's kind requires; stage is 0..(stages-1) (2 for MLPs, 3 for ATTN).
 * The stage reads its input from the plan's intermediate buffer when it is a
 * consumer stage. */
cs_status cs_chain_forward_stage(cs_chain_t plan, const void* args, int stage, void* stream);

/* After the caller has synchronised the stream: CS_OK, or the device error the
 * last forward calls recorded (CS_ERR_TIMEOUT / CS_ERR_WATCHDOG).  Blocking. */
cs_status cs_chain_status(cs_chain_t plan);

/* Zero the semaphores, counters, epoch and error word (blocking).  Required
 * after a device error before the plan runs again. */
cs_status cs_chain_reset(cs_chain_t plan);

/* Thread-local, human-readable reason for the last non-CS_OK status. */
const char* cs_last_error_string(void);

/* Sizes and device pointers of a plan, for tests and tools. */
typedef struct cs_chain_info {
  int stages;              /* 2 (MLP) or 3 (ATTN) */
  int m_tiles;             /* ceil(M/128) */
  int n_tiles[3];          /* column tiles of each stage's output */
  int units[3];            /* 128-row-block x column-tile units of each stage (semaphores) */
  int n_units;             /* schedule entries of a fused forward */
  int num_sms;             /* persistent grid size */
  int smem_bytes;          /* dynamic shared memory per CTA */
  int lag;                 /* schedule lag actually used (groups) */
  int group_m;             /* rasterisation group actually used (tile rows) */
  int tile_n[3];           /* output columns per tile of each stage */
  int tile_m;              /* rows per GEMM tile actually used (128 or 256) */
  int sched_units[3];      /* schedule entries of each stage (tiles x K-splits) */
  int split_k[3];          /* K-splits of each stage */
  int stride;              /* strided-policy stride actually used */
  void* intermediate[2];   /* H (MLP) or QKV, O (ATTN): device pointers owned by the plan */
  size_t sem_words[2];     /* length of each boundary's tile-semaphore array */
  int policy;              /* cs_policy the plan runs (AUTO resolved) */
  int tuned_entry;         /* index of the tuning-table entry applied, -1 = none */
  /* desc.out_release: device uint32 arrays of the output Y (NULL otherwise).
   * out_tile_sems[m_tiles * n_tiles[stages-1]] (128-row block-major) count the
   * forwards that stored each Y tile; out_row_sems[m_tiles] count the Y tiles
   * stored in each 128-row block, n_tiles[stages-1] per forward.  After the
   * e-th forward (e = the epoch cs_chain_debug_read_sems reports), a block of
   * rows is complete once its counter is >= e * n_tiles[stages-1]; the
   * counters are zeroed by cs_chain_reset only. */
  uint32_t* out_tile_sems;
  uint32_t* out_row_sems;
  size_t out_sem_words;    /* length of out_tile_sems */
  int sk_tiles;            /* Stream-K tail actually used: tiles of the last stage, */
  int sk_units;            /* units sharing their K-slices (0: none),               */
  int sk_q;                /* K-slices per unit (the last one may hold fewer)       */
  int workers;             /* units the grid runs at once: CTAs, or clusters of
                              tile_m / 128 CTAs that can be resident together (a
                              GPC whose SM count is not a multiple of the cluster
                              size leaves SMs out); cs_chain_plan_info, which needs
                              no GPU, reports num_sms / (tile_m / 128)          */
  int kv_chunk;            /* ATTN: key groups per attention piece (0: whole rows) */
  int raster;              /* order actually used: 1 column-major, 2 row-major,
                              3 K-range-major split consumers (desc.raster)    */
} cs_chain_info;

cs_status cs_chain_query(cs_chain_t plan, cs_chain_info* info);

/* Host-only: the geometry fields of cs_chain_info (stages .. tuned_entry) that
 * cs_chain_plan would give a plan of this desc on a device of num_sms SMs, with
 * the loaded tuning table applied; the pointer and semaphore fields are zero.
 * Needs no GPU. */
cs_status cs_chain_plan_info(const cs_chain_desc* desc, int num_sms, cs_chain_info* info);

/* What this build of the library contains (bit flags).
 *  CS_FEATURE_CLUSTER_MULTICAST: 512-row tiles, whose two CTA pairs share every
 *  weight box by TMA multicast inside a 4-CTA cluster (tile_m = 512, and the
 *  automatic choice for large M).  The package ships two builds of this ABI:
 *  libcs_chain.so has it; libcs_chain_nomc.so, the replica build that a process
 *  sharing a node with other GPUs' ranks loads, is compiled without any
 *  multicast load, refuses tile_m = 512 (CS_ERR_UNSUPPORTED), ignores
 *  tuning-table entries that name it and never picks it automatically. */
#define CS_FEATURE_CLUSTER_MULTICAST 1
int cs_library_features(void);

/* Host-only: the dispatch order a plan with this desc and grid size would use.
 * Each entry encodes one unit as (stage << 30) | (k_split << 26) | (m_tile << 14) |
 * n_tile, m_tile counting tile_m-row tiles; for an ATTN stage n_tile is the head;
 * k_split 15 marks Stream-K unit n_tile of the last stage (desc.sk_tiles).  Row blocks are taken in groups of group_m; a
 * stage's units of one group are listed column-tile-major; at step t, stage s
 * lists group t - s*lag, so every producer a unit waits on is listed before it.  *n_out receives the count; entries beyond cap
 * are not written (cap may be 0 to query the count).  Needs no GPU. */
cs_status cs_schedule_build(const cs_chain_desc* desc, int num_sms, uint32_t* units, size_t cap,
                            size_t* n_out);

/* Tuning table. ------------------------------------------------------------ */
/* Per-shape tuning of the plan's automatic choices (Flux summary, idea I4: one
 * kernel code base auto-tuned per GPU and environment).  A process-wide table
 * of measured best choices, applied by cs_chain_plan and cs_schedule_build to
 * descs that leave them on auto (see cs_chain_desc.tuned).
 *
 * File format (JSON, written by the package's tuner, consumer_gemm_chain_gb300.tune):
 *   {"format": "cs_chain_tuning", "version": 1, "entries": [ENTRY, ...], ...}
 *   ENTRY = {"kind": "gelu"|"swiglu"|"attn", "dtype": "f16"|"bf16", "H": int,
 *            "F": int, "M": int, "sms": int (grid the entry was measured on),
 *            "tile_m": 0|128|256|512, "tile_n": 0|64|128|256, "split_k": 0..15,
 *            optional "group_m": int >= 0 (default 0 = auto),
 *            optional "split_k_first": 0..15 (default 0 = as split_k),
 *            optional "raster": 0..3 (applied when the desc leaves raster on 0;
 *            default 0 = the built-in order),
 *            optional "sk_tiles": 0..65534, "sk_units": 0..16383 (Stream-K
 *            tail, applied when the desc leaves both on 0; default 0 = none),
 *            optional "layout": "kn"|"nk"|"any", "policy": "tile"|"row"|
 *            "strided"|"stream"|"any" (default any), "us": time per chain (> 0)}
 * Other keys are ignored.  Matching: entries of the same kind, dtype, H, F and
 * sms whose layout and policy fit the desc; of those, the ones at the measured
 * M nearest to desc.M on a log2 scale (ties: the smaller M); among those, for
 * policy AUTO the smallest "us", otherwise the entry naming the most of layout
 * and policy, then the smallest "us", then the first in the file. */

/* Replace the table with the entries of a JSON file.  On any error (unreadable
 * file, bad JSON, missing or out-of-range field: the message names the entry)
 * the table is left as it was.  *n_entries (may be NULL) receives the count.
 * Thread-safe; plans made earlier keep their choices. */
cs_status cs_tune_load(const char* path, int* n_entries);

/* Empty the table (the built-in rules then decide every auto field). */
cs_status cs_tune_clear(void);

/* Entries in the table. */
int cs_tune_size(void);

/* Host-only: the index of the entry a plan with this desc on num_sms SMs would
 * apply, or -1 (into *entry); *resolved (may be NULL) receives the desc with the
 * entry applied and policy AUTO resolved.  Needs no GPU. */
cs_status cs_tune_match(const cs_chain_desc* desc, int num_sms, int* entry, cs_chain_desc* resolved);

/* Testing aids. ------------------------------------------------------------ */

/* Copy boundary b's tile semaphores (b = 0: stage0->stage1, b = 1: stage1->stage2;
 * b = stages - 1: the output Y of a plan made with desc.out_release) to
 * host[0..n), then the boundary's row counters after them (m_tiles words).
 * *epoch receives the number of completed forwards.  Blocking. */
cs_status cs_chain_debug_read_sems(cs_chain_t plan, int boundary, uint32_t* host, size_t n,
                                   uint32_t* epoch);

/* Stall producer units before they release: ns[u] nanoseconds for producer unit
 * u = m_tile * n_tiles + n_tile of `stage` (at most 10 ms each).  ns = NULL or
 * n = 0 clears.  Blocking copy. */
cs_status cs_chain_debug_set_delays(cs_chain_t plan, int stage, const uint32_t* ns, size_t n);

/* Make producer unit `unit` of `stage` skip its semaphore release (-1 clears), so
 * that a consumer waiting on it times out: the bounded-wait path, without any
 * GPU fault.  The next forward then returns its error via cs_chain_status(). */
cs_status cs_chain_debug_skip_release(cs_chain_t plan, int stage, int unit);

/* Blocking device-to-device copy of plan-owned intermediate `which` (0: H or QKV,
 * 1: O) into caller device memory dst; bytes must not exceed the buffer's size
 * (M * F * 2 for H and O, M * 3F * 2 for QKV).  For stage-by-stage parity tests. */
cs_status cs_chain_debug_copy_intermediate(cs_chain_t plan, int which, void* dst, size_t bytes);

/* Enqueue on `stream` a fill of plan-owned scratch with all-ones bytes (NaN as
 * fp16, bf16 and fp32): which = 0: H or QKV, 1: O, 2: the split-K partial
 * tiles of every stage, -1: all of them.  A forward overwrites each of them
 * before any consumer may read it, so a consumer that read a K-slice before
 * its producer released it would turn its output NaN: the delay-injection
 * tests fill before every delayed forward. */
cs_status cs_chain_debug_poison_intermediate(cs_chain_t plan, int which, void* stream);

/* Blocking: set the plan's epoch to `epoch` and every counter to the value it
 * has after `epoch` forwards, modulo 2^32 (tile semaphores = epoch, row
 * counters = epoch * tiles per row block, split-K arrival counters = epoch *
 * splits, and the output counters of desc.out_release alike), so that a test
 * can run forwards across the 2^32 wrap of the epoch-counted semaphores. */
cs_status cs_chain_debug_set_epoch(cs_chain_t plan, uint32_t epoch);

/* Allocation-free MLP forward.  The pages have no counterpart to this call.
 *
 * Some callers may not allocate device memory: code running inside another
 * framework whose caching allocator owns the GPU's memory budget (a raw
 * cudaMalloc there can fail or fragment that pool), and latency-critical loops
 * where cudaMalloc/cudaFree would implicitly synchronise the device.  For them,
 * this call runs the same fused MLP chain as cs_chain_plan + cs_mlp_forward
 * without making a plan: the intermediate H, the semaphores, the control block
 * and the schedule live in one statically sized device array of
 * CS_NOALLOC_SCRATCH_BYTES (32 MiB) inside this library, which every GPU that
 * loads the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * desc: as for cs_chain_plan (kind MLP_GELU or MLP_SWIGLU), except that tiles
 * are never split along K (split_k 0 runs unsplit tiles; split_k > 1 is refused
 * with CS_ERR_UNSUPPORTED), the tuning table is not consulted (policy AUTO runs
 * TILE) and out_release is refused.  args and stream: as for cs_mlp_forward;
 * the caller still owns and passes X, the weights, b1 and Y.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call then enqueues two kernels on `stream`: a small one that
 * clears the semaphores and counters and writes the schedule into the array
 * (nothing is copied from host memory), and the chain.  So results never
 * depend on an earlier call, but the array is shared by every call on the
 * device: calls that overlap on the GPU (other streams, other threads) race
 * and must not be issued.  A shape whose intermediate, semaphores and schedule
 * need more than the array holds is rejected with CS_ERR_INVALID_ARG before any
 * work is enqueued (M * F * 2 bytes must stay well below 32 MiB).  Device-side
 * errors: read them with cs_noalloc_status() after synchronising. */
#define CS_NOALLOC_SCRATCH_BYTES (32u << 20)
cs_status cs_mlp_forward_noalloc(const cs_chain_desc* desc, const cs_mlp_args* args, void* stream);

/* Device error word of the last cs_mlp_forward_noalloc call on the current
 * device (blocking read): CS_OK, CS_ERR_TIMEOUT or CS_ERR_WATCHDOG. */
cs_status cs_noalloc_status(void);

/* Per-unit timeline: enable = 1 allocates (cudaMalloc) and zeroes a trace buffer
 * that every later forward of this plan overwrites; 0 frees it.  Each record is
 * 8 uint64: [0] unit | dispatch index << 32, [1] SM id | CTA << 16 | pair rank << 31,
 * then globaltimer ns at [2] claim, [3] dependencies published, [4] first and
 * [5] last TMA load, [6] accumulator complete, [7] epilogue done (0 = not reached).
 * Record r belongs to dispatch index r / (tile_m / 128). */
cs_status cs_chain_debug_trace(cs_chain_t plan, int enable);

/* Copy up to n records of the trace to host (8 uint64 each); *n_out = records. */
cs_status cs_chain_debug_read_trace(cs_chain_t plan, uint64_t* host, size_t n, size_t* n_out);

/* ABI version of the loaded library (CS_ABI_VERSION). */
int cs_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CS_CHAIN_H */
