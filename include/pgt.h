/*
 * pgt.h - C ABI of the GB300 (sm_103a) persistent tiled GEMM and persistent add.
 *
 * The operations follow three public pull-request pages on persistent tile scheduling:
 *   [WS]  "Work Stealing Scheduler Kernel" (ROCm/tritonBLAS PR #65): a preamble that
 *         preallocates reusable per-group int32 tile counters (MatmulConfig /
 *         matmul_preamble), a matmul entry point with a work_stealing switch whose grid is
 *         the SM count, counters reset before each launch.
 *   [TS]  "[Feature] Introduce tile scheduler" (tile-ai/tilelang PR #2441),
 *         gemm_mxfp8_blockscaled_1d1d.py: persistent 2-CTA MXFP8 GEMM with one E8M0 scale
 *         per 1 x 128 K slice, swizzled tile-id -> (m_idx, n_idx) decode with group_size
 *         and bx = m_idx * cluster_size + cta_id, warp roles fed by a stage ring.
 *   [PK]  "Implement persistent kernels" (pytorch-labs/helion PR #238): persistent_blocked
 *         and persistent_interleaved program-id loops over SM-count programs, the L2
 *         grouping decode, and the persistent elementwise add simple_add(x, y).
 *
 * Conventions for every call:
 *   - Pointers named d_* / A, B, C, x, y, out, workspace are DEVICE pointers on the
 *     context's device; pointers named h_* are HOST pointers.  The caller owns all of
 *     them and keeps them alive until the stream work has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Every compute call only enqueues work; none synchronises unless stated.
 *   - Calls return PGT_OK or a negative PGT_ERR_* status; nothing is thrown across the
 *     ABI.  Arguments are validated on the host before anything is enqueued; an invalid
 *     call enqueues nothing.
 *   - No compute call allocates device memory.  Only pgt_preamble allocates (the
 *     context's counters and error word) and pgt_destroy frees them.
 *   - Every device-side wait in these kernels is bounded (about one second).  A wait
 *     that runs out makes the kernel record PGT_ERR_TIMEOUT in the context's error word
 *     and return early; read it with pgt_last_error.
 */
#ifndef PGT_H
#define PGT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status codes */
#define PGT_OK 0
#define PGT_ERR_ARG (-1)         /* null pointer, size out of range, bad enum value */
#define PGT_ERR_ALIGN (-2)       /* base pointer or row stride not a multiple of 16 bytes */
#define PGT_ERR_UNSUPPORTED (-3) /* valid arguments the library has no kernel for */
#define PGT_ERR_CUDA (-4)        /* a CUDA runtime/driver call failed */
#define PGT_ERR_TIMEOUT (-5)     /* a device-side bounded wait ran out (from pgt_last_error) */
#define PGT_ERR_GROUPS (-6)      /* ws_groups outside [1, max_groups] of the context */
#define PGT_ERR_WORKSPACE (-7)   /* workspace missing or smaller than pgt_gemm_workspace_bytes */
#define PGT_ERR_CAPACITY (-8)    /* a trace buffer is too small for the visits it must hold */

/* ---------------------------------------------------------------------- enums */
/* Operand type.  PGT_BF16: A, B bf16.  PGT_MXFP8: A, B are OCP E4M3FN bytes with one
 * E8M0 scale byte per row and 128-wide K block ([TS] "Blockscale size: (1, 1, 128)"). */
#define PGT_BF16 0
#define PGT_MXFP8 1

/* Storage of B.  KN: K x N row-major (C = A . B literally, [WS] strides stride_bk,
 * stride_bn).  NK: N x K row-major, i.e. K contiguous ([TS] transpose_B). */
#define PGT_B_KN 0
#define PGT_B_NK 1

/* Tile scheduler modes.
 *   BLOCKED:           worker p visits tiles [p*B, min((p+1)*B, T)), B = ceil(T/P),
 *                      linear decode m = t mod m_tiles, n = t div m_tiles ([PK]).
 *   INTERLEAVED:       worker p visits p, p+P, p+2P, ... with the linear decode ([PK]).
 *   SWIZZLED:          interleaved waves (tile = P*w + p, [TS]) with the group_size
 *                      column-group decode and 2-CTA pairing ([TS]).
 *   WORK_STEALING:     tiles handed out through per-group atomic counters; G counters,
 *                      worker p homed on group p mod G, each group owning a share of the
 *                      tiles in proportion to its home workers (PGT_WS_RANGES /
 *                      PGT_WS_STRIPED below); a worker starts at its home group and
 *                      steals from the following groups ([WS]); tiles decoded like
 *                      SWIZZLED (linear when group_size == 1).  G = min(ws_groups, P):
 *                      every group has a home worker, as on the page, where the groups
 *                      (XCDs) are far fewer than the workers (CUs).  Worker p's first
 *                      tile is ticket p div G of its home group, assigned at launch (a
 *                      group's counter then hands out tickets from its number of home
 *                      workers on, and still starts each launch at zero); later tickets
 *                      are taken by a thread of the worker beside its loading thread, a few
 *                      pipeline stages before the next tile is needed.
 *                      With T <= P every ticket is assigned at launch and no counter is
 *                      touched.  P at most 65535 (PGT_ERR_ARG otherwise).
 *   BLOCKED_GROUPED_M: blocked order with the L2-grouping decode, bands of group_size
 *                      tile rows ([PK] "PERSISTENT BLOCKED WITH L2 GROUPING").
 * P is the number of persistent workers (CTAs, or CTA pairs for 2-CTA kernels) and
 * T the number of output tiles; see pgt_gemm_plan. */
#define PGT_BLOCKED 0
#define PGT_INTERLEAVED 1
#define PGT_SWIZZLED 2
#define PGT_WORK_STEALING 3
#define PGT_BLOCKED_GROUPED_M 4
/*   LAUNCH_CONTROL:    dynamic scheduling done by the hardware (Blackwell cluster launch
 *                      control; not on the pages, the GB300 counterpart of the atomic
 *                      counters): one worker is launched per tile; a running worker takes
 *                      its own tile, then asks the hardware to cancel a worker that has not
 *                      started yet and takes that worker's tile, until none is left.  Tiles
 *                      decoded like SWIZZLED.  P = T (num_workers must be 0 or T). */
#define PGT_LAUNCH_CONTROL 5

/* GEMM kernel configurations (output tile per worker, CTAs per worker).
 *   1CTA_128x128 / 1CTA_128x256: one CTA, tcgen05 cta_group::1, M=128 MMAs.
 *   2CTA_256x128 / 2CTA_256x256: a CTA pair (cluster of 2) with cta_group::2 M=256
 *   MMAs, each CTA holding 128 rows of A and half of B's tile ([TS] 2-CTA kernel).
 *   2CTA_256x224: MXFP8 only (bf16 returns PGT_ERR_UNSUPPORTED).  A pair tile 224 columns
 *   wide (a cta_group::2 MMA takes N in steps of 32), so that two fp32 accumulators and
 *   the scale columns fit in tensor memory together, and the epilogue of one tile
 *   overlaps the next tile's MMAs.  The 256x256 MXFP8 tile has room for one accumulator
 *   only.
 * PGT_CFG_AUTO picks the fastest configuration the library has for the dtype. */
#define PGT_CFG_AUTO 0
#define PGT_CFG_1CTA_128x128 1
#define PGT_CFG_1CTA_128x256 2
#define PGT_CFG_2CTA_256x128 3
#define PGT_CFG_2CTA_256x256 4
#define PGT_CFG_2CTA_256x224 5

/* Epilogue options ([WS] passes a_scale / b_scale "if quantized" and marks bias TODO).
 * Reading taken here: per-tensor scales fold into one factor alpha = a_scale * b_scale and
 * the bias is one fp32 value per output column, so C = alpha * (A . B) + bias[n], computed
 * in fp32 (one fused multiply-add per element) before the bf16 rounding. */
#define PGT_EPI_ALPHA 1
#define PGT_EPI_BIAS 2

/* pgt_preamble flags */
#define PGT_FLAG_HOST_RESET 1 /* reset work-stealing counters with a memset before every
                                 launch ([WS] reset_tile_counter) instead of in-kernel */

/* Visit-record fields written by traced launches (int32 each). */
#define PGT_VISIT_FIELDS 4 /* tile_id, m_idx, n_idx, smid */

/* Which tiles each work-stealing counter group owns (ticket j of group g is its j-th tile).
 * n_g = P div G + (g < P mod G) workers are homed on group g, S_g = n_0 + ... + n_{g-1}.
 *   RANGES:  the contiguous range [floor(T*S_g/P), floor(T*S_{g+1}/P)), a share in
 *            proportion to n_g; [g*T/G, (g+1)*T/G) when G divides P ([WS]: one counter per
 *            XCD, the XCDs holding equal numbers of CUs, each XCD with its own L2 working on
 *            its own region).
 *   STRIPED: the tiles t with (t mod P) mod G == g, in increasing order: those the workers
 *            homed on g would visit in the INTERLEAVED order (g, g+G, g+2G, ... when G
 *            divides P).  Every group advances along the same front of the decode order,
 *            so the tiles in flight are the ones a static schedule would run at that time.
 *            This suits a GPU whose L2 all SMs share.  Counters, homes, stealing, release
 *            and reset are the same. */
#define PGT_WS_RANGES 0
#define PGT_WS_STRIPED 1

typedef struct pgt_ctx pgt_ctx;

/* Full description of one GEMM C = A . B.  Leading dimensions are in elements; 0 means
 * packed (lda = K, ldb = N for KN or K for NK, ldc = N).  Row strides in bytes and the
 * base pointers of A, B and C must be multiples of 16 (TMA). */
typedef struct pgt_gemm_desc {
    int64_t M, N, K;
    int64_t lda, ldb, ldc;
    int32_t dtype;       /* PGT_BF16 | PGT_MXFP8 */
    int32_t b_layout;    /* PGT_B_KN | PGT_B_NK (MXFP8 requires NK) */
    int32_t sched_mode;  /* PGT_BLOCKED .. PGT_BLOCKED_GROUPED_M */
    int32_t group_size;  /* >= 1; swizzle / grouped-M group width in tiles */
    int32_t ws_groups;   /* work-stealing counter groups, 1 .. max_groups (0 = min(8, max)) */
    int32_t kernel_cfg;  /* PGT_CFG_* */
    int32_t num_workers; /* persistent workers; 0 = one per SM (pair), capped at T */
    int32_t epilogue;    /* 0, or PGT_EPI_ALPHA | PGT_EPI_BIAS */
    float alpha;         /* with PGT_EPI_ALPHA: C = alpha * (A . B) [+ bias] */
    int32_t ws_layout;   /* PGT_WS_RANGES | PGT_WS_STRIPED (work stealing only) */
    const float* bias;   /* with PGT_EPI_BIAS: DEVICE fp32[N], added to every row of C */
} pgt_gemm_desc;

/* What a GEMM launch will do; filled by pgt_gemm_plan. */
typedef struct pgt_gemm_plan_info {
    int32_t kernel_cfg;      /* resolved PGT_CFG_* */
    int32_t bm, bn, bk;      /* CTA tile rows, tile columns, K per pipeline stage */
    int32_t cluster_size;    /* CTAs per worker (1 or 2) */
    int32_t stages;          /* shared-memory pipeline depth */
    int32_t m_blocks;        /* ceil(M / bm) */
    int32_t n_blocks;        /* ceil(N / bn) */
    int32_t m_tiles;         /* ceil(m_blocks / cluster_size): worker-tile rows */
    int32_t tiles;           /* T = m_tiles * n_blocks */
    int32_t workers;         /* P */
    int32_t ctas;            /* P * cluster_size */
    int32_t k_iters;         /* ceil(K / bk) */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t ws_groups;       /* work-stealing counter groups in use: min(ws_groups, workers) */
} pgt_gemm_plan_info;

/* Optional launch trace (all DEVICE pointers, caller-owned).
 *   visits:   [ctas][max_visits][PGT_VISIT_FIELDS] int32, one record per tile visited,
 *             in visit order: tile_id, m_idx (worker-tile row), n_idx, SM id.
 *   counts:   [ctas] int32, number of tiles each CTA visited (may exceed max_visits;
 *             records past max_visits are dropped).
 *   times_ns: [ctas][2] int64, %globaltimer at the CTA's start and end (may be NULL). */
typedef struct pgt_trace {
    int32_t* visits;
    int64_t max_visits;
    int32_t* counts;
    int64_t* times_ns;
} pgt_trace;

/* --------------------------------------------------------------- context */
/* Create a context on `device` ([WS] MatmulConfig / matmul_preamble): queries the SM
 * count and allocates the work-stealing counters (max_groups int32 counters, each on its
 * own 128-byte line, all zero), a done counter and the device error word.
 * max_groups in [1, 64].  flags: PGT_FLAG_*.  Makes `device` current.  On success *out
 * holds the context; on failure *out is NULL. */
int pgt_preamble(int device, int max_groups, int flags, pgt_ctx** out);

/* Free a context (synchronises its device first).  NULL is accepted. */
int pgt_destroy(pgt_ctx* ctx);

/* Cooperative release of work-stealing workers ([WS] commits "Changing to one live flag per
 * XCD" and "Request CU release from the scheduler kernel", which spin on host memory; this
 * is a bounded rework).  Copies n flags (host int32, nonzero = release) into the context's
 * per-group device flags with cudaMemcpyAsync on `stream` — which may differ from the
 * stream of a running GEMM, so a release can land mid-launch.  A WORK_STEALING worker
 * reads its home group's flag (no spinning) before each ticket it would take from a counter
 * (the read is issued one decision ahead, so a raised flag takes effect within a tile) and,
 * if it is raised, takes no further tiles; the other workers steal what is left, so the
 * output is complete and identical.  A worker released before launch still runs the one
 * tile it is assigned at launch.  Group 0 is never released (its workers always finish).  Flags
 * stay raised until cleared by another call; static modes ignore them.  Until this is first
 * called on a context, its work-stealing launches do not read the flags at all.  n in
 * [1, max_groups]; pinned host memory keeps the copy asynchronous. */
int pgt_set_release(pgt_ctx* ctx, const int32_t* h_flags, int n, void* stream);

/* SM count of the context's device, or a negative status for a NULL context. */
int pgt_num_sms(const pgt_ctx* ctx);

/* Counter groups the context was created with, or a negative status. */
int pgt_max_groups(const pgt_ctx* ctx);

/* Read and clear the device error word: synchronises `stream`, then returns PGT_OK, or
 * PGT_ERR_TIMEOUT if a kernel's bounded wait ran out since the last call.  If detail is
 * not NULL it receives 4 ints: code, role (0 producer, 1 MMA, 2 epilogue, 3 scheduler),
 * block index, wait site. */
int pgt_last_error(pgt_ctx* ctx, void* stream, int32_t* detail);

/* Self-test of the bounded-wait path every kernel uses.  Launches one thread that waits on
 * an mbarrier through the same bounded wait as the GEMM roles.  arrive != 0: the thread
 * arrives first and the wait completes at once.  arrive == 0: nothing ever arrives, the
 * wait gives up after the time limit (about one second), records PGT_ERR_TIMEOUT in the
 * error word (role 3, site 12) and the kernel returns; pgt_last_error then reports it and
 * the context stays usable.  Nothing faults, traps or hangs. */
int pgt_wait_probe(pgt_ctx* ctx, int arrive, void* stream);

/* Human-readable name of a status code (static storage). */
const char* pgt_strerror(int status);

/* ------------------------------------------------------------------- GEMM */
/* Bytes of workspace pgt_gemm_ex needs for `desc` (0 for bf16).  MXFP8 needs room for the
 * scales repacked into the tensor-memory copy layout.  Returns 0 and sets nothing on
 * invalid input. */
size_t pgt_gemm_workspace_bytes(const pgt_gemm_desc* desc);

/* Resolve the kernel configuration and launch geometry for `desc` without launching.
 * Returns the same status pgt_gemm_ex would return for argument errors. */
int pgt_gemm_plan(const pgt_ctx* ctx, const pgt_gemm_desc* desc, pgt_gemm_plan_info* out);

/* C = A . B with fp32 accumulation, bf16 output rounded to nearest even.
 *   A: M x K row-major (lda), bf16 or E4M3FN bytes.
 *   B: K x N (PGT_B_KN) or N x K (PGT_B_NK) row-major (ldb), same type as A.
 *   sfa: MXFP8 only, M x (K/128) row-major E8M0 bytes, packed; sfb likewise N x (K/128).
 *        Must be NULL for bf16.
 *   C: M x N row-major bf16 (ldc).  Rows/columns past M/N are never written.
 *   workspace: device scratch of at least pgt_gemm_workspace_bytes(desc) bytes (may be
 *        NULL when that is 0); its contents are clobbered.
 *   trace: NULL, or buffers for a traced launch (a slower kernel variant that records
 *        every visit; used to check the schedule and the tail idle time).
 * Every output element is reduced over K in the same order whatever the scheduler, so for
 * one kernel_cfg the result is bit-identical across sched_mode, group_size, ws_groups,
 * ws_layout and num_workers.  (bf16 tiles of alternate waves walk K backwards.  A tile's
 * direction follows from its position and from how many workers the GPU holds at once,
 * so results can differ in the last bit between GPUs with different SM counts.)  Work
 * stealing uses the context's counters: one work-stealing launch per context may be in
 * flight at a time. */
int pgt_gemm_ex(pgt_ctx* ctx, const pgt_gemm_desc* desc, const void* A, const void* B,
                const uint8_t* sfa, const uint8_t* sfb, void* C, void* workspace,
                size_t workspace_bytes, const pgt_trace* trace, void* stream);

/* The flat form of the entry point ([WS] matmul(a, b, c, ..., work_stealing), with the
 * counter-group count of MatmulConfig): packed leading dimensions, PGT_CFG_AUTO, one worker
 * per SM (pair), contiguous counter ranges.  ws_groups: work-stealing counter groups,
 * 1 .. max_groups of the context, 0 = min(8, max_groups); a value outside [0, 64] returns
 * PGT_ERR_GROUPS before anything else is checked, one above the context's max_groups
 * returns PGT_ERR_GROUPS too.  Other arguments as in pgt_gemm_ex. */
int pgt_gemm(pgt_ctx* ctx, const void* A, const void* B, const uint8_t* sfa,
             const uint8_t* sfb, void* C, int64_t M, int64_t N, int64_t K, int dtype,
             int b_layout, int sched_mode, int group_size, int ws_groups, void* workspace,
             size_t workspace_bytes, void* stream);

/* End-to-end GEMM from host memory: copies h_A, h_B (and h_sfa, h_sfb for MXFP8) into the
 * caller's device buffers d_A, d_B, d_sfa, d_sfb with cudaMemcpyAsync, runs pgt_gemm_ex
 * into d_C, and copies d_C back to h_C, all on `stream`.  Host buffers should be pinned
 * for the copies to be asynchronous.  Device buffers use the leading dimensions of
 * `desc`; host buffers are packed copies of the same rows. */
int pgt_gemm_host(pgt_ctx* ctx, const pgt_gemm_desc* desc, const void* h_A, const void* h_B,
                  const uint8_t* h_sfa, const uint8_t* h_sfb, void* h_C, void* d_A,
                  void* d_B, uint8_t* d_sfa, uint8_t* d_sfb, void* d_C, void* workspace,
                  size_t workspace_bytes, void* stream);

/* -------------------------------------------------------------------- add */
/* out = x + y elementwise in fp32 (round to nearest even, subnormals kept), over a
 * rows x cols matrix with row strides ldx, ldy, ldo (elements; 0 = cols) ([PK]
 * simple_add).  Persistent: P workers loop over tile_r x tile_c tiles in
 * sched_mode PGT_BLOCKED or PGT_INTERLEAVED with the linear decode (tile rows fastest).
 * tile_r in [1, 1024], tile_c in [1, 4096], tile_r * tile_c <= 65536; tile_r = tile_c = 0
 * selects the wide vectorised tile.  num_workers 0 = every CTA that fits on the GPU at
 * once, or, for tiles narrower than a 128-byte line, the largest count that fits and keeps
 * the tile columns sharing a line in flight together (see pgt_add_workers).  Each worker
 * streams several of its tiles at once.  out may alias x or y exactly; other overlaps are
 * undefined.  The result does not
 * depend on the tile, the order or the worker count.  trace as in pgt_gemm_ex (m_idx /
 * n_idx are tile row / column). */
int pgt_add(pgt_ctx* ctx, const float* x, const float* y, float* out, int64_t rows,
            int64_t cols, int64_t ldx, int64_t ldy, int64_t ldo, int sched_mode, int tile_r,
            int tile_c, int num_workers, const pgt_trace* trace, void* stream);

/* Workers pgt_add will launch for these arguments (after defaults), or a negative status.
 * The default for tiles narrower than 128 bytes: with tile rows fastest a worker walks down
 * a column of tiles, and the rest of each line belongs to the neighbouring tile columns, so
 * the count is chosen to have those read at the same time (blocked: n_tiles * j workers, j
 * dividing the tile rows, each covering an equal part of one column, as many as fit at once;
 * interleaved: a multiple of tile rows * tile columns per line, up to twice what fits);
 * otherwise every CTA that fits.  Workers beyond the CTAs that fit at once run in turn on
 * the resident CTAs (CTA b runs workers b, b + grid, ...). */
int pgt_add_workers(const pgt_ctx* ctx, int64_t rows, int64_t cols, int tile_r, int tile_c,
                    int sched_mode, int num_workers);

/* ----------------------------------------------------- fused multi-space loop */
/* One elementwise tile space: out = scale * x over a rows x cols fp32 matrix (row strides
 * ldx, ldo in elements; 0 = cols).  out may alias x exactly. */
typedef struct pgt_scale_space {
    const float* x; /* DEVICE */
    float* out;     /* DEVICE */
    int64_t rows, cols, ldx, ldo;
    float scale;
    int32_t reserved;
} pgt_scale_space;

#define PGT_MAX_SPACES 8

/* Several independent tile spaces fused into ONE persistent launch ([PK] the two multi-loop
 * listings, which compute result1 = 2 * x and result2 = 3 * y): the spaces' tile ids are
 * laid end to end, P workers walk them in sched_mode PGT_BLOCKED or PGT_INTERLEAVED order,
 * and each id is decoded inside its own space with tile rows fastest.  Tiles are
 * tile_r x tile_c (both 0 = the wide 8 x 1024 tile; limits as in pgt_add).  n_spaces in
 * [1, PGT_MAX_SPACES]; num_workers 0 = every CTA that fits, capped at the tile count.
 * Traced launches record tile id, m, n, and (space << 24 | SM id) per visit.  Each output
 * is one IEEE fp32 multiply per element, whatever the order. */
int pgt_multi_loop(pgt_ctx* ctx, const pgt_scale_space* spaces, int n_spaces, int sched_mode,
                   int tile_r, int tile_c, int num_workers, const pgt_trace* trace, void* stream);

/* ----------------------------------------------------------- schedule log */
/* Run only the device tile scheduler (the same code the GEMM kernels run) over an
 * m_blocks x n_blocks grid of CTA tiles with `cluster_size` CTAs per worker, and record
 * each worker's visits in `trace` (one record list per WORKER, not per CTA).  One
 * single-thread worker per block; num_workers >= 1, and for PGT_LAUNCH_CONTROL exactly the
 * tile count (one worker per tile; cancelled workers record nothing).  Work stealing uses
 * the context's counters and release flags like the GEMM, with ws_layout a PGT_WS_* and
 * min(ws_groups, num_workers) counter groups (num_workers at most 65535, PGT_ERR_ARG
 * otherwise). */
int pgt_schedule_log(pgt_ctx* ctx, int64_t m_blocks, int64_t n_blocks, int cluster_size,
                     int sched_mode, int group_size, int ws_groups, int ws_layout, int num_workers,
                     const pgt_trace* trace, void* stream);

/* ------------------------------------------------------ allocation-free GEMM */
/* No counterpart in the pages: an addition for callers that cannot allocate device memory
 * (code running inside another runtime's memory-pool or allocator hook, plugins whose
 * device memory is budgeted up front, real-time paths that forbid allocation after
 * start-up).  They cannot create a context, because pgt_preamble allocates.
 *
 * C = A . B in bf16 with the WORK_STEALING scheduler, exactly as pgt_gemm_ex computes it
 * (same kernel, so the same bits), on the CURRENT device, with packed leading dimensions
 * and PGT_CFG_AUTO.  The scratch the kernel needs (ws_groups tile counters, a done counter
 * and an error word) is a fixed 2304-byte file-scope __device__ array that every GPU which
 * loads the library holds until the process exits; no call allocates or frees anything.
 *   A, B, C, M, N, K, b_layout, group_size: as in pgt_gemm (bf16 only).
 *   ws_groups: 1 .. PGT_NOALLOC_MAX_GROUPS (0 = 8); larger values return PGT_ERR_GROUPS.
 *   d_err: NULL, or a caller-owned DEVICE int32[4] the kernel writes if a bounded wait
 *          runs out (code, role, block, site); this call does not clear it.  With NULL a
 *          timeout only lands in a line of the shared array, which the next call clears and
 *          no call reads: the call still returns PGT_OK and C may be incomplete.  Callers
 *          that must detect a timeout pass d_err and read it after the stream finishes.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current; make that first call before any stream capture.  A first
 * call made while `stream` is capturing returns PGT_ERR_ARG and enqueues nothing.  Every call
 * clears the counters on `stream` before its launch.  All calls share the one array per
 * device: calls that overlap on the GPU (different streams, or graph replays running
 * concurrently) race on it and give wrong results. */
#define PGT_NOALLOC_MAX_GROUPS 16
int pgt_gemm_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                     int b_layout, int group_size, int ws_groups, int32_t* d_err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PGT_H */
