/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE routing + dispatch + grouped-GEMM
 * library (libmoe_gb300.so).
 *
 * The operation is the "MoE Dispatch + GEMM" fused kernel of mKernel, as the
 * articles "Conozca mKernel: una biblioteca de nucleo fusionado ..."
 * (7minutos.es) and its Arabic twin (k7ail.com) describe it in their table of
 * the five fused kernels, row "MoE Dispatch + GEMM": route MoE tokens to
 * their expert ranks (an all-to-all), and run the per-expert grouped GEMM in
 * the same kernel, on tokens as soon as they land, with no round trip through
 * a staging buffer.  The same articles, section on the design properties,
 * describe the kernel as persistent, with CTAs that assign themselves roles
 * and a per-shape number of SMs per role.  On one GPU the all-to-all becomes
 * a scatter into R simulated per-rank receive buffers in local HBM.
 *
 * Notation: T tokens, d hidden width (GEMM K), E experts, k experts per
 * token, N expert output width, R simulated expert ranks, S = T*k routed
 * slots.  bf16 tensors are passed as uint16_t bit patterns.
 *
 * Conventions shared by every call
 *  - Ownership: the caller allocates and owns every device buffer and the
 *    stream.  The library owns only the host-side plan object.  No call
 *    allocates device memory, synchronises the host, or copies device data
 *    to the host, except moe_read_status (documented there).
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Calls are asynchronous and stream-ordered.  Calls that
 *    share one workspace must be ordered on one stream; overlapping them on
 *    the GPU is a race.
 *  - Alignment: x, W, Y and the receive buffers 16-byte aligned; int32 and
 *    fp32 arrays 4-byte aligned; the workspace 256-byte aligned.  All rows
 *    are dense (row stride = width).  A misaligned pointer is
 *    MOE_ERR_INVALID_ARG (MOE_ERR_WORKSPACE for the workspace).
 *  - Errors: argument errors are returned synchronously, before any launch,
 *    and leave every buffer untouched.  Errors found on the device (a bounded
 *    wait that gave up, a receive buffer overflow) are written into the
 *    caller's `dev_status` buffer and read later with moe_read_status.  No
 *    kernel traps.
 *  - Shape limits: 1 <= E <= 1024; 1 <= k <= min(E, 32); 0 <= T; T*k < 2^31;
 *    d % 16 == 0 and 16 <= d <= 65536; N % 16 == 0 and 16 <= N; E % R == 0
 *    and 1 <= R <= 32.  Outside them: MOE_ERR_UNSUPPORTED.  (A reduction d
 *    that is not a multiple of 64 ends in a shorter last k-block: its MMAs
 *    stop at d.)
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, bad field   */
    MOE_ERR_UNSUPPORTED = 2,  /* valid arguments outside the library's shape limits */
    MOE_ERR_WORKSPACE = 3,    /* workspace missing or misaligned                      */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (or no device)     */
    MOE_ERR_TIMEOUT = 5,      /* device: a bounded wait for a ready flag gave up      */
    MOE_ERR_CAPACITY = 6,     /* device: a rank's receive buffer is too small         */
    MOE_ERR_DEVICE = 7        /* device: an internal pipeline wait gave up            */
} moe_status_t;

/* moe_shape_t.route_flags.  The expert choice is the same under every flag;
 * only the gate weights differ.  RENORM alone is Mixtral-style gating (the
 * softmax over the k chosen logits); SIGMOID | RENORM with a selection bias
 * (moe_route_biased) is DeepSeek-V3-style gating. */
#define MOE_ROUTE_RENORM 1
#define MOE_ROUTE_SIGMOID 2

/* Opaque host-side plan: shape, tile configuration and role split. */
typedef struct moe_plan_s* moe_plan_t;

typedef struct moe_shape {
    int32_t T;                  /* tokens                                               */
    int32_t d;                  /* hidden width = GEMM reduction length                */
    int32_t E;                  /* experts                                              */
    int32_t k;                  /* experts per token                                    */
    int32_t N;                  /* expert output width                                  */
    int32_t num_ranks;          /* R simulated expert ranks; 0 means 1                  */
    int32_t rank_capacity_rows; /* rows in each rank's receive buffer; 0 means T*k      */
    int32_t tile_n;             /* GEMM tile width: 0 = auto, else 128, 192 or 256;
                                   512 with CTA pairs only (tile_m 0 or 256, N >= 512)  */
    int32_t producer_ctas;      /* CTAs that start in the scatter role: 0 = all of them */
    int32_t num_ctas;           /* persistent grid size: 0 = one CTA per SM             */
    int64_t timeout_ns;         /* limit of every device-side wait: 0 = 2 s             */
    int32_t debug_skip_publish; /* fault injection: 0 = off; m > 0 = never publish the
                                   ready flag of m-tile m-1 (the consumer's bounded wait
                                   then reports MOE_ERR_TIMEOUT)                         */
    int32_t route_flags;        /* how moe_route scores the picks (gates); 0 = softmax
                                   over all E logits.  MOE_ROUTE_SIGMOID: logistic of
                                   each logit instead; MOE_ROUTE_RENORM: each token's k
                                   gates divided by their sum.  Other bits must be 0.   */
    int32_t tile_m;             /* GEMM tile height: 0 = auto; 128 = one CTA per tile;
                                   256 = CTA pairs (tcgen05 cta_group::2; needs N >= 256
                                   and tile_n 0 or 256)                                  */
    int32_t out_dtype;          /* element type of Y: MOE_OUT_F32 (0, default) or
                                   MOE_OUT_BF16 (fp32 accumulation rounded once to bf16,
                                   nearest even)                                         */
} moe_shape_t;

/* moe_shape_t.out_dtype */
#define MOE_OUT_F32 0
#define MOE_OUT_BF16 1

typedef struct moe_plan_info {
    int32_t tile_m, tile_n, tile_k;   /* GEMM tile (rows, columns, reduction step); rows =
                                         256 when CTA pairs share each tile                */
    int32_t stages;                   /* shared-memory pipeline depth                   */
    int32_t num_ctas, producer_ctas;  /* persistent grid and its initial scatter role   */
    int32_t sm_count;                 /* SMs of the plan's device                       */
    int32_t smem_bytes;               /* dynamic shared memory of the fused kernel      */
    int32_t max_mtiles;               /* upper bound on 128-row tiles: floor(S/128) + E */
    int32_t route_blocks;             /* CTAs of the routing kernel                     */
    int64_t workspace_bytes;          /* size moe_plan reported                         */
    int32_t half_tiles;               /* 1: a moe_dispatch_gemm / moe_grouped_gemm /
                                         moe_gather_gemm schedule of at most num_ctas/2
                                         tiles runs each tile as two half-width tiles
                                         (the same bits; single-CTA plans of tile_n 128
                                         or 256); 0: whole tiles only                   */
    int32_t background_scatter;       /* CTA-pair plans, moe_dispatch_gemm: > 0 when every
                                         warp scatters only the rows of the first experts
                                         (those holding this many pair tiles) before the
                                         GEMM and warp 3 of each CTA copies the rest beside
                                         it (layers of N >= 8192); 0: the whole scatter
                                         first.  Same bits either way                     */
} moe_plan_info_t;

/*
 * moe_plan -- validate a shape and build a plan for `device`.
 *   shape            in:  the layer shape and optional tuning fields.
 *   device           in:  CUDA device ordinal the plan (and every later call)
 *                         runs on; it must be current when calls are made.
 *   plan             out: the new plan; release it with moe_plan_destroy.
 *   workspace_bytes  out: size of the device workspace every moe_route and
 *                         moe_dispatch_gemm call of this plan needs.  The
 *                         caller allocates it, 256-byte aligned, and fills it
 *                         with zeros ONCE before the first call (and again
 *                         after any device error status); the calls return
 *                         their counters to zero themselves.
 * Host only (queries device attributes); launches nothing.
 * Tuning overrides read from the environment when the plan is built (for sweeps
 * and tests; none changes a result bit, and unset is the default schedule):
 *   MOE_HALF_TILES=0|2     single-CTA plans: never / always split tiles in halves
 *   MOE_BG_HEAD=n          CTA-pair plans: pair tiles the all-warps scatter covers
 *                          before the GEMM (0: the whole scatter first)
 *   MOE_SCATTER_PARTS=p    the scatter's parts per expert (1: expert-major)
 *   MOE_TILE_BAND=b        row tiles per schedule band (0: the whole expert)
 */
MOE_API moe_status_t moe_plan(const moe_shape_t* shape, int device, moe_plan_t* plan,
                      size_t* workspace_bytes);

/* Release a plan (NULL is accepted). */
MOE_API moe_status_t moe_plan_destroy(moe_plan_t plan);

/* Copy the plan's chosen configuration into *info. */
MOE_API moe_status_t moe_plan_info(moe_plan_t plan, moe_plan_info_t* info);

/*
 * moe_route -- the routing half of "MoE Dispatch + GEMM": choose each
 * token's experts and lay out the destination rows.
 *   logits   in:  fp32 [T][E] router logits (any bias already added); finite.
 *   topk_idx out: int32 [T][k]; slot j holds the expert with the (j+1)-th
 *                 largest logit; between equal logits the lower expert index
 *                 comes first (-0.0 equals +0.0).
 *   topk_w   out: fp32 [T][k]; the gate of each pick, from the chosen logit
 *                 l: exp(l - max) / sum over all E of exp(logit - max) (default)
 *                 or 1 / (1 + exp(-l)) (MOE_ROUTE_SIGMOID in the shape's
 *                 route_flags); with MOE_ROUTE_RENORM each token's k gates are
 *                 then divided by their sum.  fp32 with expf; with SIGMOID |
 *                 RENORM a token whose chosen logits are all below about -87
 *                 gets NaN gates (every logistic rounds to 0).
 *   counts   out: int32 [E]; rows routed to each expert.
 *   offsets  out: int32 [E+1]; exclusive prefix sum of counts, offsets[E] = S.
 *   perm     out: int32 [S]; destination row -> source slot t*k+j.  Rows are
 *                 grouped by expert (ascending), then by token, then slot.
 *   dest     out: int32 [S]; the inverse of perm.
 *   workspace in/out: the plan's workspace (see moe_plan).
 * Launches two kernels on `stream`.  Results are identical bit for bit on
 * every run (no atomics decide any order).
 */
MOE_API moe_status_t moe_route(moe_plan_t plan, const float* logits,
                       int32_t* topk_idx, float* topk_w,
                       int32_t* counts, int32_t* offsets,
                       int32_t* perm, int32_t* dest,
                       void* workspace, void* stream);

/*
 * moe_route_biased -- moe_route with a per-expert selection bias: expert e of
 * token t is ranked by the key fp32(logits[t][e] + selection_bias[e]) instead
 * of the logit (same order rule, same tie rule), while the gates are computed
 * from the unbiased logits as moe_route describes.  This is the bias that
 * auxiliary-loss-free load balancing adjusts between steps: it moves tokens
 * between experts without entering the weights the outputs are scaled by.
 *   selection_bias in: fp32 [E] on the device, finite; NULL = moe_route.
 * Other arguments, launches and errors as for moe_route.
 */
MOE_API moe_status_t moe_route_biased(moe_plan_t plan, const float* logits,
                                      const float* selection_bias,
                                      int32_t* topk_idx, float* topk_w,
                                      int32_t* counts, int32_t* offsets,
                                      int32_t* perm, int32_t* dest,
                                      void* workspace, void* stream);

/*
 * moe_dispatch_gemm -- the fused dispatch + per-expert grouped GEMM, one
 * persistent kernel.  Scatter CTAs copy token rows into the rank receive
 * buffers and publish a ready flag per 128-row tile; GEMM CTAs wait for each
 * tile's flag and run it on the tensor cores (bf16 inputs, fp32
 * accumulation) as soon as it is ready.
 *   x        in:  bf16 [T][d] token rows.
 *   offsets  in:  int32 [E+1] from moe_route (device).
 *   perm     in:  int32 [S] from moe_route (device).
 *   W        in:  bf16 [E][d][N] expert weights (N contiguous).
 *   recv     in:  HOST array of R device pointers; recv[r] is rank r's receive
 *                 buffer, bf16 [rank_capacity_rows][d].  Rank r owns experts
 *                 [r*E/R, (r+1)*E/R); its buffer receives the destination rows
 *                 [offsets[r*E/R], offsets[(r+1)*E/R]) in order (out).
 *   Y        out: [S][N], fp32 (or bf16 with MOE_OUT_BF16 in the plan's shape);
 *                 Y[i] = recv row of destination row i times W[e(i)], where
 *                 e(i) is the expert whose segment holds i.
 *                 Row order is the destination (expert-sorted) order; undoing
 *                 the permutation is the caller's step.
 *   workspace in/out: the plan's workspace.
 *   dev_status in/out: device int32[4], zeroed by the caller before first use.
 *                 The first device-side error writes {code, tile or row,
 *                 expert, call epoch}; later errors do not overwrite it.
 * Launches one kernel on `stream`.
 */
MOE_API moe_status_t moe_dispatch_gemm(moe_plan_t plan, const uint16_t* x,
                               const int32_t* offsets, const int32_t* perm,
                               const uint16_t* W, void* const* recv, void* Y,
                               void* workspace, int32_t* dev_status, void* stream);

/*
 * moe_dispatch_gemm_combine -- moe_dispatch_gemm with the combine step (the
 * reverse exchange that the "MoE Dispatch + GEMM" row of the articles' table
 * of fused kernels implies after the per-expert GEMM) fused into the GEMM's
 * epilogue: no Y is written; each destination row i, times the gate of its
 * slot s = perm[i], goes straight into its token's output row:
 *   out[t][n] = sum_{j<k} topk_w[t][j] * (x[t] . W[topk_idx[t][j]][:, n]),
 * with each product rounded to fp32 and the terms summed in fp32 in
 * ascending expert order.  The token's lowest expert stores its term; each
 * higher expert's term is added (a 16-byte fp32 reduction) only after the
 * lower terms of that token and column tile have landed: every 128-row tile
 * publishes an epoch-tagged completion word per column tile, and a row waits
 * for the words of its token's lower rows.  Those tiles belong to lower
 * experts, which the schedule claims first, so the waits always end; the
 * order of the additions, and so every bit of `out`, does not depend on
 * timing, role split or grid size, for any k.  It differs from moe_combine's
 * fused multiply-adds by the rounding of each product.  Nothing is zeroed:
 * every element of `out` is written by its token's first term.
 * When to use it: it beats moe_dispatch_gemm + moe_combine where a token's
 * terms sit in tiles claimed far apart (k = 2 over a few large experts: about
 * 1.1-1.2x).  Where k > 2 and the experts are many, a later term's tile is
 * claimed just after the lower ones it waits for, the epilogues serialize,
 * and the separate combine is faster (1.4x at k = 4 over 64 experts, 3x at
 * k = 8 over 256).
 *   dest   in:  int32 [T*k] from moe_route (device).
 *   topk_w in:  fp32 [T][k] from moe_route (device).
 *   out    out: fp32 [T][N], 16-byte aligned.
 * Other arguments as for moe_dispatch_gemm (the receive buffers are written;
 * the plan's out_dtype does not apply).  Launches one kernel.
 */
MOE_API moe_status_t moe_dispatch_gemm_combine(moe_plan_t plan, const uint16_t* x,
                                       const int32_t* offsets, const int32_t* perm,
                                       const int32_t* dest, const float* topk_w,
                                       const uint16_t* W, void* const* recv, float* out,
                                       void* workspace, int32_t* dev_status, void* stream);

/*
 * moe_dispatch_gemm_swiglu -- moe_dispatch_gemm for a gated (SwiGLU) expert
 * up-projection.  The plan's N is 2F: W1's first F columns are the gate
 * projection and the last F the up projection.  Each GEMM tile computes the
 * gate and the up columns of the same F-columns side by side (tile_n/2 of
 * each) and its epilogue writes
 *   H[i][f] = bf16( silu(g) * u ),  g = (A_i . W1[e][:, f]),
 *                                  u = (A_i . W1[e][:, F+f]),  silu(g) = g / (1 + e^-g)
 * with g, u accumulated in fp32 and the activation in fp32, rounded once to
 * bf16 (nearest even).  The articles fix no expert activation; this entry
 * point serves Mixtral- and DeepSeek-style experts, whose down projection is
 * moe_grouped_gemm on H.
 *   W1  in:  bf16 [E][d][2F] (2F = the plan's N; F a multiple of 8).
 *   H   out: bf16 [S][F], destination order, 16-byte aligned.
 * Other arguments as for moe_dispatch_gemm.  MOE_ERR_UNSUPPORTED for a plan
 * made with tile_n = 192 (the halves must be whole 64-column boxes).
 */
MOE_API moe_status_t moe_dispatch_gemm_swiglu(moe_plan_t plan, const uint16_t* x,
                                      const int32_t* offsets, const int32_t* perm,
                                      const uint16_t* W1, void* const* recv, uint16_t* H,
                                      void* workspace, int32_t* dev_status, void* stream);

/*
 * moe_gather_gemm -- the per-expert grouped GEMM with its A rows gathered
 * straight from the token rows: for each destination row i, row x[perm[i] / k]
 * is copied from global memory into the GEMM's shared-memory tile by 16-byte
 * asynchronous copies of two warps per CTA, with no receive buffer in between (a
 * variant of moe_dispatch_gemm for one GPU, where the all-to-all has no wire
 * to cross; it measures what landing the rows in a receive buffer costs).  Y is
 * bit for bit the Y of moe_dispatch_gemm on the same plan (the same tiles; on
 * CTA pairs the peer's gathered stages are passed to the leader by a relay
 * thread).  With no scatter phase and no receive-buffer traffic it is the faster
 * of the two on one GPU where the dispatch's scatter is a large share (about
 * 20% on a fine-grained layer of 64 experts, top-4).
 *   x, offsets, perm, W, Y, workspace, dev_status, stream: as for
 *   moe_dispatch_gemm.  No receive buffers.  Launches one kernel.
 */
MOE_API moe_status_t moe_gather_gemm(moe_plan_t plan, const uint16_t* x, const int32_t* offsets,
                                     const int32_t* perm, const uint16_t* W, void* Y,
                                     void* workspace, int32_t* dev_status, void* stream);

/*
 * moe_grouped_gemm -- the per-expert grouped GEMM alone, on rows the caller
 * has already laid out in destination order (for example H from
 * moe_dispatch_gemm_swiglu, for the down projection).  Same kernel and tiles
 * as moe_dispatch_gemm with no scatter role and no ready flags.
 *   A        in:  bf16 [S][d] (the plan's d), destination order, 16-byte aligned.
 *   offsets  in:  int32 [E+1]: expert e owns rows [offsets[e], offsets[e+1]);
 *                 offsets[E] must equal S = T*k.
 *   W        in:  bf16 [E][d][N].
 *   Y        out: [S][N] in the plan's out_dtype; Y[i] = A[i] x W[e(i)].
 * Workspace and status as for moe_dispatch_gemm (the plan's workspace; a plan
 * may serve both entry points on one stream).  Launches one kernel.
 */
MOE_API moe_status_t moe_grouped_gemm(moe_plan_t plan, const uint16_t* A, const int32_t* offsets,
                                      const uint16_t* W, void* Y, void* workspace,
                                      int32_t* dev_status, void* stream);

/*
 * moe_set_trace -- per-CTA timing records of the plan's later GEMM launches
 * (moe_dispatch_gemm and its variants), for measuring the schedule: where a
 * launch's time goes between the scatter, the ready-flag waits and the GEMM.
 *   trace  in/out: device buffer of at least (SM count) x 8 uint64 (the SM count
 *                  is moe_plan_info's sm_count), 8-byte aligned; NULL turns
 *                  tracing off (the default).  Each launch overwrites record b
 *                  (words 8b .. 8b+7) of every CTA b it runs:
 *                  0 start, 1 end of its scatter share (0 if none), 2 first
 *                  tile's rows ready, 4 tiles it loaded (the halves of a split
 *                  tile count as two), 5 last load issued,
 *                  6 end (global-timer ns); 3 total ns waiting for ready flags;
 *                  7 its role ticket.
 * The records cost a few stores per tile.  Host only; no launch.
 */
MOE_API moe_status_t moe_set_trace(moe_plan_t plan, void* trace, int64_t bytes);

/*
 * moe_router_logits -- the step before the path: the router logits that
 * moe_route consumes, L = x @ W_r + bias, on the GPU.  The articles name no
 * router; this library fixes its arithmetic so that routing stays bit-exact
 * against a CPU reference: for each (token t, expert e) an fp32 accumulator
 * runs fused multiply-adds over i ascending (each bf16 x bf16 product is exact
 * in fp32), then the fp32 bias is added.  CUDA cores, no tensor cores.
 *   x      in:  bf16 [T][d].
 *   W_r    in:  bf16 [d][E] (E contiguous).
 *   bias   in:  fp32 [E] or NULL.
 *   logits out: fp32 [T][E].
 * Launches one kernel on `stream`; no workspace.
 */
MOE_API moe_status_t moe_router_logits(moe_plan_t plan, const uint16_t* x, const uint16_t* W_r,
                                       const float* bias, float* logits, void* stream);

/*
 * moe_combine -- the step after the path: undo the destination permutation and
 * weight each token's k expert outputs by its gates.  The articles' table row
 * "MoE Dispatch + GEMM" describes the dispatch side only; the combine is the
 * mirror image that completes the layer's output.
 *   Y      in:  [S][N] from moe_dispatch_gemm (destination order), fp32 or bf16
 *                as the plan's out_dtype says.
 *   topk_w in:  fp32 [T][k] from moe_route.
 *   dest   in:  int32 [S] from moe_route.
 *   out    out: fp32 [T][N]; out[t][n] = sum_{j<k} topk_w[t][j] * Y[dest[t*k+j]][n],
 *               fp32 fused multiply-adds in ascending j (identical on every run).
 * Launches one kernel on `stream`; no workspace.
 */
MOE_API moe_status_t moe_combine(moe_plan_t plan, const void* Y, const float* topk_w,
                                 const int32_t* dest, float* out, void* stream);

/*
 * moe_read_status -- synchronise `stream`, copy the 4-word device status to
 * out[4] and return out[0] as a moe_status_t (MOE_ERR_CUDA if the copy or
 * the synchronisation fails).  This is the one call that waits for the GPU.
 */
MOE_API moe_status_t moe_read_status(const int32_t* dev_status, void* stream, int32_t out[4]);

/*
 * moe_route_noalloc -- moe_route for callers that cannot allocate device
 * memory.  The pages describe no such variant; it exists for embedders that
 * are not allowed to call cudaMalloc themselves: for example a plugin inside
 * an inference server or framework that owns every byte of device memory and
 * forbids allocation after start-up, or a code path that must not fail on an
 * out-of-memory error.  It computes exactly what moe_route computes (same
 * kernels, same outputs, bit for bit) but takes no workspace: its scratch (a
 * per-CTA count table and a ticket counter) lives in a static device array
 * of 1 MiB + 256 bytes inside the library, which every GPU that loads the
 * library holds until the process exits.  Arguments as for moe_route.
 *  - Limit: ceil(T/64) * E <= 262144 (for example T = 16384 with E <= 1024,
 *    or T = 65536 with E <= 256).  A larger plan returns MOE_ERR_UNSUPPORTED
 *    before any launch.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  A lookup that fails returns MOE_ERR_CUDA and
 *    is tried again by the next call on that device.
 *  - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *    routine.  It clears the ticket counter with cudaMemsetAsync on `stream`
 *    before its launch; the count table is fully rewritten by every call.
 *  - Every call shares the one array, which keeps the last call's contents:
 *    calls that overlap on the GPU (different streams, or different host
 *    threads without ordering) race and give wrong results.
 */
MOE_API moe_status_t moe_route_noalloc(moe_plan_t plan, const float* logits,
                                       int32_t* topk_idx, float* topk_w,
                                       int32_t* counts, int32_t* offsets,
                                       int32_t* perm, int32_t* dest, void* stream);

/* Static string naming a status code. */
MOE_API const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
