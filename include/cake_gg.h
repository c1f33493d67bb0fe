/*
 * cake_gg.h -- C ABI of the GB300 (sm_103a) ragged BF16 grouped GEMM.
 *
 * The operation (flashinfer PR #8258, "perf(cake_moe_grouped_gemm): run the
 * split k512 wgrad tail whole on the least-loaded clusters", opening summary):
 * a ragged grouped GEMM for MoE expert training with BF16 inputs and FP32
 * accumulation, in three passes -- forward Y = X W^T, data gradient dX = G W,
 * weight gradient dW = G^T X -- with BF16 or FP32 output.  Expert e owns the
 * rows [offsets[e], offsets[e+1]) of X, G, Y and dX.  The dense projection
 * family (flashinfer PR #8363, "Summary" and "Definitions") is the E = 1 case.
 *
 * Layouts (row-major, last index contiguous, no padding between rows):
 *   X  [M_max, K] bf16      W  [E, N, K] bf16      G  [M_max, N] bf16
 *   Y  [M_max, N] out_dtype dX [M_max, K] out_dtype dW [E, N, K] out_dtype
 *   offsets [E+1] int32, device memory: offsets[0] == 0, non-decreasing,
 *   offsets[E] <= M_max.  Rows >= offsets[E] of Y and dX are never written;
 *   the weight gradient ignores them.  An empty expert gets an exact zero dW.
 *
 * Deterministic mode (PR #8258, opening summary: the deterministic kernel
 * gives the same bits on every run): every
 * output element is computed by a fixed sequence of FP32 operations that
 * depends only on the plan -- which cake_gg_plan() derives from (pass, E,
 * M_max, N, K, out_dtype) alone unless a plan override below is set -- and
 * the offsets: never on
 * max_sms, on which CTA runs a tile, or on arrival order (the weight
 * gradient takes its tiles from a counter at run time; the results are the
 * same bits whichever CTA computes a tile).  Split reductions add FP32
 * partials in split order and round once.  Non-deterministic mode
 * (PR #8258, opening summary, 2nd paragraph: split tail partials are added
 * into one FP32 tile by atomic reductions, and a ticket per tile tells the
 * last CTA to finish it) may change the order of the weight gradient's split
 * sums from run to run.  The forward and
 * data-gradient passes never split and are deterministic in both modes.
 *
 * Ownership: the caller owns every buffer (inputs, outputs, offsets,
 * workspace) and the plan.  The compute calls allocate nothing, free nothing,
 * launch nothing but their kernel and never synchronise the host; they
 * enqueue work on `stream` (a cudaStream_t, NULL = the legacy default stream)
 * and return.  The workspace must stay allocated and unused by anyone else
 * until the stream has run the call; calls that share one workspace must be
 * ordered on one stream.
 *
 * Workspace contents: fill the workspace with zeros once after allocating it
 * (and again after a device-detected error).  Every call that ends without a
 * device-detected error leaves it ready for the next call, so no call clears
 * it.  Split-tile tickets are tagged with a per-call number and never need
 * clearing; that number lives in the workspace header and each call's last
 * CTA advances it on the device, so a call replayed from a captured CUDA
 * graph gets a fresh number as well.  The unit counter (workspace header) is
 * zeroed by the last CTA of each call.
 *
 * Environment overrides (tuning and test hooks, unset in normal use):
 *   read by cake_gg_plan(), recorded in the plan it fills (a deterministic
 *   plan's summation order follows them):
 *     CAKE_GG_TILE_N (64..256), CAKE_GG_TILE_K (64, 128, 256), CAKE_GG_PAIR=0
 *     (single CTAs only) or 2 (pairs wherever the tile allows), CAKE_GG_WIDE (0: no 256 x 512 weight-gradient tiles,
 *     2: wherever they fit), CAKE_GG_WIDE_FD=1 (512-wide forward / data-
 *     gradient tiles), CAKE_GG_SPLIT_CHUNK (k-blocks per split, 0 = no split),
 *     CAKE_GG_CSPLIT (0: splits through workspace slots; 2..8 cluster splits,
 *     for pairs 2..4: clusters of two CTAs per split), CAKE_GG_EPI_GROUPS (1 or
 *     2 epilogue warpgroups for the forward / data gradient), CAKE_GG_TAIL=0
 *     (no split tail of either kind), CAKE_GG_NTAIL (N-split tail of 256 x 512
 *     tiles: 0 = off, the default; 1 = by its rule; 2 or 4 = that many column
 *     pieces), CAKE_GG_STREAMK (0: never, the default; 1: by the cost rule;
 *     2: wherever the walk applies), CAKE_GG_STREAMK_KB (its segment length
 *     in k-blocks), CAKE_GG_STAGES, CAKE_GG_STAGING_BUFS (1 or 2),
 *     CAKE_GG_DECIDED=0 (the non-deterministic planner ignores its table of
 *     measured points where a plan rule failed the decision protocol);
 *   read by each compute call, changing no result:
 *     CAKE_GG_PDL=0 (no programmatic dependent launch), CAKE_GG_ROUTER_STAGGER
 *     (the router's per-unit k-order stagger, default 7, 0 = in order;
 *     changes the router's summation order), CAKE_GG_DYN=0 (static
 *     unit order), CAKE_GG_SPIN_NS (an early split's poll for its tile's
 *     other partials, default 6000), CAKE_GG_PREFETCH (L2 prefetch distance
 *     in stages), CAKE_GG_STACK=0 and CAKE_GG_TMA_STORE=0 (plainer copy and
 *     store paths).
 *
 * Errors: host-detected problems return a non-zero cake_gg_status_t and
 * enqueue nothing.  Problems only the GPU can see (bad offsets, a bounded wait
 * that expired) are recorded in the workspace's status word, which keeps the
 * first such error until cake_gg_check_status() reads and resets it; the
 * kernel then skips its remaining work and returns (it never traps).  Output
 * contents are unspecified after any error.
 */
#ifndef CAKE_GG_H
#define CAKE_GG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CAKE_GG_ABI_VERSION 1

typedef enum {
    CAKE_GG_OK = 0,
    CAKE_GG_ERR_INVALID_ARG = 1,  /* null pointer, size out of range, plan/call mismatch   */
    CAKE_GG_ERR_ALIGNMENT = 2,    /* a base pointer not 16-byte aligned, or N/K not multiples of 8 */
    CAKE_GG_ERR_OVERFLOW = 3,     /* a size product overflows 64-bit or a TMA coordinate   */
    CAKE_GG_ERR_UNSUPPORTED = 4,  /* current device is not sm_103 (GB300), or a dtype is unknown */
    CAKE_GG_ERR_WORKSPACE = 5,    /* workspace missing or smaller than plan->workspace_bytes */
    CAKE_GG_ERR_CUDA = 6,         /* a CUDA runtime/driver call failed                      */
    CAKE_GG_ERR_BAD_OFFSETS = 7,  /* device-detected: offsets not 0-based, decreasing or > M_max */
    CAKE_GG_ERR_TIMEOUT = 8,      /* device-detected: a bounded wait inside the kernel expired */
    CAKE_GG_ERR_SCRATCH_LIMIT = 9 /* the problem needs more scratch than cake_gg_wgrad_noalloc's fixed maximum */
} cake_gg_status_t;

typedef enum { CAKE_GG_FWD = 0, CAKE_GG_DGRAD = 1, CAKE_GG_WGRAD = 2 } cake_gg_pass_t;
typedef enum { CAKE_GG_BF16 = 0, CAKE_GG_FP32 = 1 } cake_gg_dtype_t;

/* Plan: a caller-owned plain struct filled by cake_gg_plan(); nothing to free.
 * The first block holds the problem as given; the second holds the choices
 * made for it.  The choices are a pure function of the first block minus
 * max_sms, so max_sms changes only how many CTAs run, never a result bit.
 * With pair = 2 the launch uses clusters of two CTAs, so the number of CTAs
 * is max_sms rounded down to an even number (at least 2). */
typedef struct cake_gg_plan {
    int32_t abi_version;     /* CAKE_GG_ABI_VERSION                                 */
    int32_t pass;            /* cake_gg_pass_t                                      */
    int32_t E;               /* experts, 1 .. 1024                                  */
    int32_t N;               /* W rows per expert (output width of the forward)     */
    int32_t K;               /* W columns (reduction length of the forward)         */
    int32_t out_dtype;       /* cake_gg_dtype_t                                     */
    int64_t M_max;           /* rows allocated in X / G / Y / dX (0 .. 2^31 - 1)    */
    int32_t deterministic;   /* 1 = bitwise reproducible, 0 = split sums by atomics */
    int32_t max_sms;         /* cap on persistent CTAs; 0 = every SM of the device  */
    /* chosen by cake_gg_plan() */
    int32_t tile_m;          /* MMA rows per tile (128)                             */
    int32_t tile_n;          /* MMA columns per tile (64 .. 256)                    */
    int32_t tile_k;          /* reduction elements per pipeline stage (64, 128, 256) */
    int32_t stages;          /* shared-memory ring depth                            */
    int32_t pair;            /* 2: two CTAs compute a 256-row tile as one tcgen05 MMA,
                                each holding half of the B tile; 1: single CTAs      */
    int32_t swap_ab;         /* weight gradient: 1 = MMA rows run over K (thin N)   */
    int32_t split_chunk;     /* weight gradient: k-blocks per split, 0 = no split   */
    int32_t debug_flags;     /* test-only fault injection; 0 in normal use          */
    uint64_t timeout_ns;     /* limit of every in-kernel wait (default 2 s)         */
    uint64_t workspace_bytes;/* bytes of workspace the compute call needs           */
    int32_t staging_bufs;    /* epilogue staging buffers per warp (1 or 2)          */
    int32_t cluster_splits;  /* weight gradient: >0 = that many splits per tile run as
                                one cluster (of CTAs, or of pairs: 2 CTAs per split)
                                and reduce on chip (no workspace partials)          */
    int32_t tail_units;      /* weight gradient: the last tail_units units of the walk */
    int32_t tail_splits;     /* are each split into tail_splits pieces whose FP32
                                partials are summed in split order (0 = no tail split) */
    int32_t streamk_kblocks; /* weight gradient of one expert: > 0 = stream-K walk, the
                                work cut into segments of this many k-blocks that cross
                                tile boundaries; a tile's pieces are summed in k order */
    int32_t epi_groups;      /* forward / data gradient: 2 = a second epilogue warpgroup
                                takes every other tile (short reductions); else 1 */
    int32_t tail_nsplit;     /* weight gradient of 256 x 512 pair tiles: > 1 = the last
                                tail_units units run as that many column pieces each,
                                every piece over all k-blocks (no partials; the bits
                                of the whole units); 0 = none                       */
    int32_t reserved[1];
} cake_gg_plan_t;

/* Debug flag (tests only): the CTA that takes the walk's first unit (its even
 * CTA, in a pair) arms its first pipeline stage but issues no copy into it, so
 * the consumer's bounded wait expires and the call reports
 * CAKE_GG_ERR_TIMEOUT through the status word. */
#define CAKE_GG_DEBUG_DROP_FIRST_LOAD 1

/* Fill *plan for one pass.  Pure host arithmetic: no CUDA call, no allocation.
 * Checks E in [1, 1024], N, K >= 1 and multiples of 8 (16-byte rows for the
 * tensor-memory-access engine), M_max in [0, 2^31 - 1], out_dtype and pass,
 * and that every byte size fits in 64 bits.  max_sms < 0 is invalid. */
int cake_gg_plan(cake_gg_plan_t *plan, int pass, int32_t E, int64_t M_max, int32_t N,
                 int32_t K, int out_dtype, int deterministic, int32_t max_sms);

/* Forward Y = X W_e^T per expert (PR #8258 opening summary).  X, W, Y,
 * offsets: device pointers, 16-byte aligned.  out_dtype and deterministic
 * must equal the plan's.  Writes rows [0, offsets[E]) of Y only. */
int cake_gg_fwd(const cake_gg_plan_t *plan, const void *X, const void *W, void *Y,
                const int32_t *offsets, int out_dtype, int deterministic,
                void *workspace, size_t workspace_bytes, void *stream);

/* Data gradient dX = G W_e per expert (PR #8258 opening summary: the input
 * gradient of the grouped expert layer; PR #8363 "Definitions" for the dense
 * family's [T, d_out] gradient and [T, d_in] result).  G [M_max, N],
 * W [E, N, K], dX [M_max, K]: device pointers, 16-byte aligned.  out_dtype and
 * deterministic must equal the plan's.  Writes rows [0, offsets[E]) of dX
 * only. */
int cake_gg_dgrad(const cake_gg_plan_t *plan, const void *G, const void *W, void *dX,
                  const int32_t *offsets, int out_dtype, int deterministic,
                  void *workspace, size_t workspace_bytes, void *stream);

/* Weight gradient dW_e = G_e^T X_e per expert, the sum over the expert's rows
 * (the ragged reduction; PR #8258 opening summary, with BF16 or FP32 dW and
 * its split tails, and PR #8363 "Definitions" for the dense family's
 * [d_out, d_in] weight gradient).  G [M_max, N], X [M_max, K], dW [E, N, K]:
 * device pointers, 16-byte aligned; every element of dW is written (zeros for
 * an empty expert).  out_dtype and deterministic must equal the plan's. */
int cake_gg_wgrad(const cake_gg_plan_t *plan, const void *G, const void *X, void *dW,
                  const int32_t *offsets, int out_dtype, int deterministic,
                  void *workspace, size_t workspace_bytes, void *stream);

/* Weight gradient without any allocation and without a caller workspace.
 *
 * The pages have no counterpart to this entry point.  It exists for callers
 * that cannot allocate device memory: a plugin or custom-operator interface
 * that hands the library only its input and output pointers and a stream
 * (no allocator, no workspace hook), and code that must not allocate once it
 * is running (an allocation can synchronise the device or fail under memory
 * pressure in the middle of a training step).
 *
 * Same arguments and result as cake_gg_wgrad() minus the workspace: the
 * library uses its own scratch, a fixed array of CAKE_GG_NOALLOC_SCRATCH_BYTES
 * in device memory that every GPU which loads the library holds until the
 * process exits.  Nothing is allocated or freed by the call.
 *  - A plan whose workspace_bytes exceeds CAKE_GG_NOALLOC_SCRATCH_BYTES is
 *    rejected with CAKE_GG_ERR_SCRATCH_LIMIT before anything is enqueued.
 *  - The first call on each device looks up the scratch array's device
 *    address (with that device current); make that first call before any
 *    stream capture begins.  The address is kept together with the context
 *    it belongs to: after a device reset (a new primary context) the next
 *    call looks it up again, so make that call before any capture as well.
 *  - Every call on a device shares the one scratch array, which keeps the
 *    last call's contents; each call clears the parts that must start at
 *    zero.  Calls whose kernels overlap on the GPU (different streams without
 *    ordering between them) race on the scratch and give wrong results:
 *    order them on one stream.
 *  - Device-detected errors are written to the scratch's status word, which
 *    callers cannot read; outputs are unspecified after such an error. */
#define CAKE_GG_NOALLOC_SCRATCH_BYTES (32u << 20)
int cake_gg_wgrad_noalloc(const cake_gg_plan_t *plan, const void *G, const void *X, void *dW,
                          const int32_t *offsets, int out_dtype, int deterministic, void *stream);

/* ---- FP32 router GEMM (BF16x3 emulation) ---------------------------------
 *
 * The dense projection family's FP32 router GEMM (flashinfer PR #8438,
 * "Summary", which names a router GEMM over 256 experts in FP32 emulated
 * with three BF16 products): logits Y [T, R] = X [T, K] W^T, with X [T, K],
 * router weights W [R, K] and Y all FP32, row-major.  The emulation (the pages name it and nothing more; the
 * usual reading is taken): every value v is split as hi = bf16(v) and
 * lo = bf16(v - hi), round to nearest even, and
 *   Y[t, r] ~= sum_k x_hi w_hi + x_hi w_lo + x_lo w_hi
 * with every product exact and the sum accumulated in FP32 by the tensor
 * cores.  It drops x_lo w_lo and the split residues:
 * |Y - X W^T| <= 3 * 2^-16 * sum_k |x_k w_k| plus FP32 accumulation error.
 *
 * The plan is a caller-owned POD; `gemm` is the plan of the kernel the call
 * runs: the grouped GEMM's forward pass in a router mode (E = 1) whose
 * converter warps split FP32 X tiles into BF16 high and low tiles on chip. */
typedef struct cake_gg_router_plan {
    int32_t abi_version;     /* CAKE_GG_ABI_VERSION                          */
    int32_t R;               /* router outputs (experts), a multiple of 8    */
    int64_t T;               /* tokens, 0 .. 2^31 - 1                        */
    int32_t K;               /* model width, a multiple of 8                 */
    int32_t reserved;
    uint64_t workspace_bytes;/* the call's whole workspace (see below)       */
    cake_gg_plan_t gemm;     /* the forward plan it runs                     */
} cake_gg_router_plan_t;

/* Fill *rp.  Pure host arithmetic.  CAKE_GG_ERR_ALIGNMENT unless R and K are
 * multiples of 8; CAKE_GG_ERR_INVALID_ARG for T < 0, R or K < 1, max_sms < 0;
 * CAKE_GG_ERR_OVERFLOW when a size does not fit.  rp->workspace_bytes is the
 * workspace the call needs: the kernel's header, the offsets of the
 * one-expert problem and W' [R, 2K] = [w_hi | w_lo] in BF16 (4 R K bytes). */
int cake_gg_router_plan(cake_gg_router_plan_t *rp, int64_t T, int32_t R, int32_t K, int32_t max_sms);

/* Y = X W^T by BF16x3 emulation.  X, W, Y, workspace: device pointers,
 * 16-byte aligned; the workspace is rp->workspace_bytes, caller-owned, filled
 * with zeros once after allocation (as for cake_gg_fwd), unused by anyone else
 * until the stream has run the call.  Enqueues two kernels on `stream` (W's
 * split into W', then the router kernel); allocates nothing, never
 * synchronises.  Host-detected errors return non-zero and enqueue nothing
 * (CAKE_GG_ERR_INVALID_ARG also for a plan whose forward plan's tile shape or
 * ring depth is not the one cake_gg_router_plan gives); the router kernel's
 * device-detected errors land in the workspace's status word
 * (cake_gg_check_status).  The split kernel is a programmatic dependent of
 * the stream's previous kernel (it waits for it before touching memory;
 * CAKE_GG_PDL=0 launches it plainly). */
int cake_gg_router_fp32(const cake_gg_router_plan_t *rp, const float *X, const float *W, float *Y,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Synchronise `stream`, return the status word of `workspace` (CAKE_GG_OK,
 * or the first _BAD_OFFSETS / _TIMEOUT recorded by a call since the last
 * check) and reset it to CAKE_GG_OK; CAKE_GG_ERR_CUDA if a CUDA call failed. */
int cake_gg_check_status(const void *workspace, void *stream);

/* Static, never-NULL description of a status code. */
const char *cake_gg_strerror(int code);

/* Measurement aid (co-run robustness): launch `ctas` CTAs on `stream`, each
 * holding one SM (it takes the maximum shared memory) for `ns` nanoseconds,
 * then exiting.  Bounded by time alone; touches no memory.  The grouped-GEMM
 * calls on another stream then run on the remaining SMs; the weight
 * gradient's tile counter lets the CTAs that do run take the whole walk.
 * CAKE_GG_ERR_INVALID_ARG for ctas outside 1..1024 or ns above 10 s. */
int cake_gg_corun_spinner(int32_t ctas, uint64_t ns, void *stream);

/* Host-side replica of the kernel's tile walk, for testing the scheduler on
 * any machine.  Given host offsets[E+1], writes up to `capacity` tiles, each
 * as 10 int32 {expert, m_tile, n_tile, split, n_splits, kblock_begin,
 * kblock_end, ticket, column_begin, column_count} (the last two: the columns
 * of the n_tile the unit computes, all tile_n of them but for an N-split
 * tail piece), in walk order (heaviest expert first for the weight
 * gradient; the order in which the CTAs take them from the tile counter, or
 * by a fixed stride), and stores the total tile count in *count.  Returns CAKE_GG_ERR_BAD_OFFSETS for offsets
 * the kernel would reject. */
int cake_gg_tile_walk(const cake_gg_plan_t *plan, const int32_t *offsets_host,
                      int64_t capacity, int32_t *tiles_out, int64_t *count);

#ifdef __cplusplus
}
#endif

#endif /* CAKE_GG_H */
