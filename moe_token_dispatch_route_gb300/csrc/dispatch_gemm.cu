// Fused dispatch + per-expert grouped GEMM: one persistent kernel.
//
// The operation is the "MoE Dispatch + GEMM" row of the mKernel articles'
// table of the five fused kernels: an all-to-all that routes token rows to
// their expert ranks, and the per-expert grouped GEMM in the same kernel,
// run on rows as soon as they land, without a staging round trip.  Their
// design section describes persistent kernels whose CTAs assign themselves
// roles, with a per-shape number of SMs per role.
//
// On one GB300 the all-to-all becomes a scatter into R per-rank receive
// buffers in local HBM.  Design:
//  * Grid = one CTA per SM (about 200 KB of shared memory each, so exactly one
//    fits), 256 threads, all resident together as in any persistent kernel.
//    Each CTA takes a ticket from a workspace counter when it starts; the
//    first `producer_ctas` tickets (by default all of them) take the scatter
//    role first.
//  * Scatter role: all 8 warps copy destination rows (perm -> token row of x)
//    into the rank buffers with 16-byte loads and stores, 4 rows per work
//    unit, in the order the GEMM consumes them.  The last unit of each
//    128-row tile publishes the tile's ready flag (release store of the call's
//    epoch).  Then the CTA joins the GEMM role.  CTA pairs on wide layers
//    (N >= 8192: few rows per second feed the GEMM) copy only the first
//    experts' rows this way, enough for the first two waves of tiles; warp 3
//    of every CTA then copies the rest through registers beside the GEMM,
//    publishing the same flags.
//  * GEMM role, warp-specialised: warp 0 lane 0 claims tiles from a
//    workspace counter (expert-major, then column tile, then row tile),
//    waits for the row tile's flag (acquire, then a generic->async proxy
//    fence) and streams A (receive rows, K-major) and B (W, N-major) through
//    a multi-stage TMA ring with 128-byte swizzle; warp 1 lane 0 issues
//    tcgen05.mma (M=128, N=tile_n, K=16; bf16 in, fp32 accumulation in
//    TMEM, two accumulators so the epilogue of one tile overlaps the next
//    tile's MMAs); warps 4-7 read the accumulator with tcgen05.ld and store
//    the valid rows and columns of Y (fp32) with streaming stores.
//  * Variants of the same kernel: a gated (SwiGLU) epilogue that writes
//    silu(gate) * up in bf16 from the two halves of a tile; a bf16 Y; a
//    grouped mode on rows already in place (no scatter, no flags); and a
//    direct-gather mode whose warps 2-3 copy A rows straight from x.
//  * Every wait is bounded (globaltimer).  A ready flag that never comes is
//    reported as MOE_ERR_TIMEOUT and the tile is computed anyway, so the
//    pipeline stays consistent; a pipeline wait that gives up reports
//    MOE_ERR_DEVICE and all roles leave through the same teardown (drain of
//    issued TMA loads and MMAs, TMEM release).  The last CTA to finish resets
//    the workspace counters and records the epoch.
#include <cuda_bf16.h>

#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kMaxStages = 8;
constexpr int kEpiWarp0 = 4;  // warps 4..7: TMEM lane quarters 0..3

struct TileInfo {
    int e, m, n, mtile;
    int row0;  // global destination row of the tile's first row
    int rows;  // valid rows 1..128; -1 marks the end of the schedule
    int rank;
    int arow;  // first row inside the rank's receive buffer
    int m128;  // CTA pairs: 1 for an expert's last tile of at most 128 rows, run as an
               // M=128 pair MMA (64 rows per CTA); 0 otherwise
    int half;  // single CTAs: 0 the whole tile; 1 / 2 its left / right half of the columns
               // (small schedules run every tile as two halves)
};

constexpr int kMaxPieceBufs = 8;

// One staged piece of a destination row (scatter role): where it goes and
// which 16-byte vectors of the row it holds.
struct PieceRec {
    uint16_t* dst;  // destination row in the rank buffer
    int q0, q1;     // vector range [q0, q1) of the row
    int e, j;       // expert and unit inside the expert
    int flags;      // 1: row valid, 2: last piece of the unit
    int pad;
};

struct SmemCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t afull[kMaxStages];  // gather mode, peer CTA of a pair: its gather warps' rows landed
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t sfull[kRing];
    uint64_t sempty[kRing];
    uint64_t mma_done;
    TileInfo ring[kRing];
    uint32_t tmem_base;
    int abort;
    int role;
    uint32_t epoch;
    int wsum[kThreads / 32];
    PieceRec piece[kThreads / 32][kMaxPieceBufs];  // scatter: per-warp ring of staged pieces
};

static_assert(sizeof(TileInfo) % 8 == 0, "tile descriptions move in 8-byte asynchronous stores");
static_assert(offsetof(SmemCtl, ring) % 8 == 0, "ring slots must be 8-byte aligned");

struct Waiter {
    volatile int* abort;
    int32_t* status;
    long long flag_timeout_ns;  // ready-flag waits
    long long pipe_timeout_ns;  // pipeline mbarrier waits (generous: they may include a flag wait)
    uint32_t epoch;
};

// Trace stamps (moe_set_trace): one record of kTraceWords per CTA, written by
// one thread each; nothing is written when the trace is off.
__device__ __forceinline__ void trace_set(const DispatchGemmParams& p, int word, unsigned long long v) {
    if (p.trace) p.trace[(size_t)blockIdx.x * kTraceWords + word] = v;
}
__device__ __forceinline__ void trace_add(const DispatchGemmParams& p, int word, unsigned long long v) {
    if (p.trace) p.trace[(size_t)blockIdx.x * kTraceWords + word] += v;
}

// Bounded mbarrier wait.  Returns false if the CTA is aborting or the wait
// exceeded the timeout (then it reports MOE_ERR_DEVICE and starts the abort).
__device__ bool wait_bar(uint32_t bar, uint32_t parity, const Waiter& w, int where,
                         bool honor_abort = true, bool cluster_scope = false) {
    auto poll = [&]() {
        return cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (poll()) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (poll()) return true;
        if ((i & 127u) == 0) {
            if (honor_abort && *w.abort) return false;
            if (global_timer_ns() - t0 > (uint64_t)w.pipe_timeout_ns) {
                report_error(w.status, kStDevice, where, -1, (int)w.epoch);
                *w.abort = 1;
                return false;
            }
        }
    }
}

// Bounded wait for a row tile's ready flag.  On timeout the error is
// reported and the caller proceeds (the tile's result is then undefined).
__device__ void wait_flag(const uint32_t* flag, const Waiter& w, int mtile, int e) {
    if (ld_acquire_gpu(flag) == w.epoch) return;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ld_acquire_gpu(flag) == w.epoch) return;
        if ((i & 31u) == 0) {
            if (*w.abort) return;
            if (global_timer_ns() - t0 > (uint64_t)w.flag_timeout_ns) {
                report_error(w.status, kStTimeout, mtile, e, (int)w.epoch);
                return;
            }
        }
    }
}

// Exclusive prefix table[0..nch E] (nch E <= 1024) of per-(chunk, expert) counts, all
// threads.  With U_e = ceil(count_e / div), entry c E + e counts the part
// [floor(c U_e / nch), floor((c+1) U_e / nch)) of expert e's U_e items: chunk-major
// order, nch = 1 giving the per-expert ceil(count / div) prefix.
__device__ void build_expert_table(const int32_t* offsets, int E, int div, int* table, int* wsum, int nch = 1) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int base = tid * 4;
    const int n = nch * E;
    int loc[4];
    int sum = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = base + u;
        int v = 0;
        if (i < n) {
            const int c = i / E, e = i - c * E;
            const int cnt = __ldg(offsets + e + 1) - __ldg(offsets + e);
            const long long U = (cnt + div - 1) / div;
            v = (int)((c + 1) * U / nch - c * U / nch);
        }
        loc[u] = v;
        sum += v;
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int pre = 0, total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
        if (w < warp) pre += wsum[w];
        total += wsum[w];
    }
    int run = pre + incl - sum;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        if (base + u < n) table[base + u] = run;
        run += loc[u];
    }
    if (tid == 0) table[n] = total;
    __syncthreads();
}

// largest e in [0, E) with table[e] <= u (u < table[E]); empty experts are skipped
__device__ __forceinline__ int expert_of(const int* table, int E, int u) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (table[mid] <= u) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Scatter role: all 8 warps of a scatter CTA copy token rows into the rank
// receive buffers.
//
// Work unit = up to 4 consecutive destination rows of one expert inside one
// 128-row tile; only non-empty units exist.  Units are visited strided over all
// scatter warps of all scatter CTAs in chunk-major order: each expert's units are
// cut into p.nch equal parts (unit_base holds the prefix over (part, expert)), and
// part c of every expert comes before part c+1 of any.  An expert's rows are in token
// order, so part c of every expert holds about the same c-th slice of the tokens,
// and the k copies of a token row are read while its x row is still in L2 (one DRAM
// read per token row instead of up to k).  Each row is split into pieces of at most
// 512 16-byte vectors.
//
// The loads are cp.async.cg (global -> shared, no L1 allocation) into a
// lane-private staging area carved from the idle GEMM stage buffers (24 KB
// per warp, split into 3-8 piece buffers), so the number of bytes in flight
// is set by shared memory rather than by the small L1 left beside it.  A
// warp keeps up to nbuf-1 pieces loading while it drains the oldest one
// (shared -> registers -> global).  Each piece's destination is kept in a
// per-warp ring in shared memory, so the drain needs no lookups.  After every
// four finished units (and at the end) lane 0 fences, cumulative over the
// warp's stores through __syncwarp, and counts the units in; the last unit of
// a tile releases the tile's ready flag with the call's epoch.
constexpr int kWarpSlotsPerLaneMax = 48;  // 48 x 16 B per lane = 24 KB per warp

// 16-byte staging slots per lane that fit in a stage area of `bytes` (8 warps x 32 lanes)
constexpr int scatter_slots_per_lane(size_t bytes) {
    return (int)(bytes / ((kThreads / 32) * 32 * 16)) < kWarpSlotsPerLaneMax
               ? (int)(bytes / ((kThreads / 32) * 32 * 16))
               : kWarpSlotsPerLaneMax;
}
constexpr int kPieceVecsMax = 512;
constexpr int kPublishBatch = 4;  // finished units per fence + publication

// The warp's walk over its units (c, c + stride, c + 2 stride, ...).  The
// units' metadata is fetched 32 units at a time, one unit per lane, so the
// dependent loads (offsets, then perm) cost one round trip per 32 units rather
// than one per unit; the current unit's fields are broadcast from its lane.
struct UnitCursor {
    int c, stride, total;  // current unit (lane-uniform)
    int slot;              // lane holding the current unit's metadata
    bool done;
    // current unit, lane-uniform
    int e, j, nrows, rank;
    int r, q;              // row of the unit and piece of the row
    // this lane's unit of the batch
    int m_e, m_j, m_nrows, m_rank;
    int m_tok[kRowsPerChunk];    // token of each row (-1: skip the row)
    int m_local[kRowsPerChunk];  // row inside the rank buffer
};

__device__ void cursor_fetch_batch(UnitCursor& u, const DispatchGemmParams& p, const int* unit_base,
                                   uint32_t epoch, int lane) {
    const int c = u.c + lane * u.stride;
    u.m_nrows = 0;
    u.m_e = u.m_j = u.m_rank = 0;
#pragma unroll
    for (int r = 0; r < kRowsPerChunk; ++r) {
        u.m_tok[r] = -1;
        u.m_local[r] = -1;
    }
    if (c >= u.total) return;
    const int i = expert_of(unit_base, p.nch * p.E, c);  // (part, expert) holding unit c
    const int part = i / p.E;
    const int e = i - part * p.E;
    const int seg0 = __ldg(p.offsets + e);
    const int cnt = __ldg(p.offsets + e + 1) - seg0;
    const long long U = (cnt + kRowsPerChunk - 1) / kRowsPerChunk;
    const int j = (int)(part * U / p.nch) + (c - unit_base[i]);  // unit index inside the expert
    const int e_per_rank = p.E / p.R;
    const int rank = e / e_per_rank;
    const int rbase = __ldg(p.offsets + rank * e_per_rank);
    const int nrows = min(kRowsPerChunk, cnt - j * kRowsPerChunk);
    u.m_e = e;
    u.m_j = j;
    u.m_rank = rank;
    u.m_nrows = nrows;
    int perm_v[kRowsPerChunk];
#pragma unroll
    for (int r = 0; r < kRowsPerChunk; ++r)
        perm_v[r] = r < nrows ? __ldg(p.perm + seg0 + j * kRowsPerChunk + r) : 0;
#pragma unroll
    for (int r = 0; r < kRowsPerChunk; ++r) {
        if (r >= nrows) continue;
        const int row = seg0 + j * kRowsPerChunk + r;
        const int local = row - rbase;
        const int tok = perm_v[r] / p.k;
        if (local >= p.cap) {
            report_error(p.status, kStCapacity, row, rank, (int)epoch);
        } else if (tok < 0 || tok >= p.T) {
            report_error(p.status, kStDevice, -3, row, (int)epoch);
        } else {
            u.m_tok[r] = tok;
            u.m_local[r] = local;
        }
    }
}

__device__ void cursor_select(UnitCursor& u) {
    u.done = u.c >= u.total;
    u.e = __shfl_sync(kFull, u.m_e, u.slot);
    u.j = __shfl_sync(kFull, u.m_j, u.slot);
    u.nrows = __shfl_sync(kFull, u.m_nrows, u.slot);
    u.rank = __shfl_sync(kFull, u.m_rank, u.slot);
    u.r = 0;
    u.q = 0;
}

// first unit of the walk
__device__ void cursor_init(UnitCursor& u, const DispatchGemmParams& p, const int* unit_base, int first,
                            int stride, int total, uint32_t epoch, int lane) {
    u.c = first;
    u.stride = stride;
    u.total = total;
    u.slot = 0;
    cursor_fetch_batch(u, p, unit_base, epoch, lane);
    cursor_select(u);
}

// next unit of the walk
__device__ void cursor_next(UnitCursor& u, const DispatchGemmParams& p, const int* unit_base,
                            uint32_t epoch, int lane) {
    u.c += u.stride;
    if (++u.slot == 32) {
        u.slot = 0;
        cursor_fetch_batch(u, p, unit_base, epoch, lane);
    }
    cursor_select(u);
}

// token and rank-buffer row of row r of the current unit (lane-uniform)
__device__ __forceinline__ void cursor_row(const UnitCursor& u, int r, int& tok, int& local) {
    int t = u.m_tok[0], l = u.m_local[0];
#pragma unroll
    for (int i = 1; i < kRowsPerChunk; ++i)
        if (r == i) {
            t = u.m_tok[i];
            l = u.m_local[i];
        }
    tok = __shfl_sync(kFull, t, u.slot);
    local = __shfl_sync(kFull, l, u.slot);
}

// Counts `n` finished units in (their rows already written and fenced by the
// caller).  The per-tile counters are incremented first, all n together, so
// their round trips overlap; the unit that completes a tile then releases the
// tile's ready flag with the call's epoch and returns the counter to zero.
__device__ void publish_units(const DispatchGemmParams& p, const int* mt_base, const int* es,
                              const int* js, int n, uint32_t epoch) {
    uint32_t prev[kPublishBatch];
    int mtile[kPublishBatch], units[kPublishBatch];
#pragma unroll
    for (int i = 0; i < kPublishBatch; ++i) {
        if (i >= n) break;
        const int cnt = __ldg(p.offsets + es[i] + 1) - __ldg(p.offsets + es[i]);
        const int m = js[i] / kChunksPerTile;
        mtile[i] = mt_base[es[i]] + m;
        units[i] = min(kChunksPerTile, (cnt + kRowsPerChunk - 1) / kRowsPerChunk - m * kChunksPerTile);
        prev[i] = atomicAdd(p.chunk_cnt + mtile[i], 1u);
    }
#pragma unroll
    for (int i = 0; i < kPublishBatch; ++i) {
        if (i >= n) break;
        if (prev[i] + 1u == (uint32_t)units[i]) {
            __threadfence();
            p.chunk_cnt[mtile[i]] = 0u;  // ready for the next call
            fence_proxy_async_global();
            if (mtile[i] != p.skip_publish) st_release_gpu(p.flags + mtile[i], epoch);
        }
    }
}

// `slots_per_lane` 16-byte slots per lane of staging (at least 32, so that every warp has at
// least two piece buffers), all inside the stage area
__device__ void scatter_role(const DispatchGemmParams& p, const int* mt_base, const int* unit_base,
                             int role, uint32_t epoch, uint8_t* staging, SmemCtl* ctl,
                             int slots_per_lane, int end_units) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = p.producer_ctas * (kThreads / 32);
    const int nvec = p.d / 8;
    const int piece_vecs = min(nvec, kPieceVecsMax);
    const int pieces_per_row = (nvec + piece_vecs - 1) / piece_vecs;
    const int lane_slots = (piece_vecs + 31) / 32;  // 1..16
    const int nbuf = min(kMaxPieceBufs, slots_per_lane / lane_slots);  // >= 1 when slots >= 16
    const uint32_t wslots = smem_addr(staging) + (uint32_t)(warp * slots_per_lane * 32 * 16);
    PieceRec* ring = ctl->piece[warp];

    UnitCursor L;
    cursor_init(L, p, unit_base, role * (kThreads / 32) + warp, nwarps, end_units, epoch, lane);

    int pend_e[kPublishBatch], pend_j[kPublishBatch];
    int npend = 0;
    long long gi = 0, gd = 0;  // pieces issued, pieces drained
    for (;;) {
        // keep up to nbuf - 1 pieces loading
        while (!L.done && gi - gd < nbuf - 1) {
            const int b = (int)(gi % nbuf);
            int tr, lr;
            cursor_row(L, L.r, tr, lr);
            const int q0 = L.q * piece_vecs;
            const int q1 = min(q0 + piece_vecs, nvec);
            if (tr >= 0) {
                const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)tr * p.d);
                for (int i = 0; i < lane_slots; ++i) {
                    const int v = q0 + lane + 32 * i;
                    if (v < q1)
                        cp_async16_cg(wslots + (uint32_t)(((b * lane_slots + i) * 32 + lane) * 16), src + v);
                }
            }
            cp_async_commit();  // one group per piece (empty for a skipped row)
            const bool last = L.q == pieces_per_row - 1 && L.r == L.nrows - 1;
            if (lane == 0) {
                PieceRec rec;
                rec.dst = tr >= 0 ? p.recv[L.rank] + (size_t)lr * p.d : nullptr;
                rec.q0 = q0;
                rec.q1 = q1;
                rec.e = L.e;
                rec.j = L.j;
                rec.flags = (tr >= 0 ? 1 : 0) | (last ? 2 : 0);
                rec.pad = 0;
                ring[b] = rec;
            }
            ++gi;
            if (++L.q == pieces_per_row) {
                L.q = 0;
                if (++L.r == L.nrows) cursor_next(L, p, unit_base, epoch, lane);
            }
        }
        if (gd == gi) break;
        // the oldest piece: wait for this lane's part, then store it
        cp_async_wait_dyn((int)(gi - gd - 1));
        __syncwarp();
        const int b = (int)(gd % nbuf);
        const PieceRec rec = ring[b];
        if (rec.flags & 1) {
            uint4* dst = reinterpret_cast<uint4*>(rec.dst);
            for (int i = 0; i < lane_slots; ++i) {
                const int v = rec.q0 + lane + 32 * i;
                if (v < rec.q1) {
                    uint4 t;
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(t.x), "=r"(t.y), "=r"(t.z), "=r"(t.w)
                                 : "r"(wslots + (uint32_t)(((b * lane_slots + i) * 32 + lane) * 16)));
                    dst[v] = t;
                }
            }
        }
        ++gd;
        if (rec.flags & 2) {
            pend_e[npend] = rec.e;
            pend_j[npend] = rec.j;
            ++npend;
        }
        if (npend == kPublishBatch || (L.done && gd == gi && npend > 0)) {
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) {
                __threadfence();
                publish_units(p, mt_base, pend_e, pend_j, npend, epoch);
            }
            npend = 0;
        }
    }
    cp_async_wait<0>();
    // the staging area becomes TMA (async-proxy) destination again
    fence_proxy_async_smem();
}

// Background scatter (one warp of a CTA, beside the GEMM roles): the units
// [first, total) in steps of `stride`, each row copied through registers with
// kBgVecs 16-byte loads per lane in flight, then stored; finished units are
// counted in and their tiles' flags released exactly as the all-warps scatter does.
constexpr int kBgVecs = 16;
__device__ void scatter_background(const DispatchGemmParams& p, const int* mt_base, const int* unit_base,
                                   int first, int stride, int total, uint32_t epoch) {
    const int lane = threadIdx.x & 31;
    const int nvec = p.d / 8;
    UnitCursor L;
    cursor_init(L, p, unit_base, first, stride, total, epoch, lane);
    int pend_e[kPublishBatch], pend_j[kPublishBatch];
    int npend = 0;
    while (!L.done) {
        int tr[kRowsPerChunk], lr[kRowsPerChunk];
#pragma unroll
        for (int r = 0; r < kRowsPerChunk; ++r) {
            tr[r] = -1;
            lr[r] = 0;
            if (r < L.nrows) cursor_row(L, r, tr[r], lr[r]);
        }
        uint16_t* rbuf = p.recv[L.rank];
        const int items = L.nrows * nvec;
        for (int f0 = 0; f0 < items; f0 += 32 * kBgVecs) {
            uint4 t[kBgVecs];
#pragma unroll
            for (int i = 0; i < kBgVecs; ++i) {
                const int f = f0 + lane + 32 * i;
                const int r = f / nvec;
                int tok = -1;
#pragma unroll
                for (int q = 0; q < kRowsPerChunk; ++q)
                    if (r == q) tok = tr[q];
                if (f < items && tok >= 0)
                    t[i] = ld_nc_na_v4(reinterpret_cast<const uint4*>(p.x + (size_t)tok * p.d) + (f - r * nvec));
            }
#pragma unroll
            for (int i = 0; i < kBgVecs; ++i) {
                const int f = f0 + lane + 32 * i;
                const int r = f / nvec;
                int tok = -1, loc = 0;
#pragma unroll
                for (int q = 0; q < kRowsPerChunk; ++q)
                    if (r == q) {
                        tok = tr[q];
                        loc = lr[q];
                    }
                if (f < items && tok >= 0)
                    reinterpret_cast<uint4*>(rbuf + (size_t)loc * p.d)[f - r * nvec] = t[i];
            }
        }
        pend_e[npend] = L.e;
        pend_j[npend] = L.j;
        ++npend;
        cursor_next(L, p, unit_base, epoch, lane);
        if (npend == kPublishBatch || (L.done && npend > 0)) {
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) {
                __threadfence();
                publish_units(p, mt_base, pend_e, pend_j, npend, epoch);
            }
            npend = 0;
        }
    }
}

// Epilogue staging: each epilogue warp turns a 32-row x 32-column fp32 block (one row per
// lane, as tcgen05.ld 32x32b returns it) into row-contiguous 128-byte segments through a
// padded shared-memory tile, so every store instruction writes 4 rows x 128 B instead of
// 32 partial lines.  The row stride of 36 floats keeps the 16-byte writes and reads free
// of bank conflicts.
constexpr int kEpiStride = 36;
constexpr int kEpiWarpFloats = 32 * kEpiStride;
constexpr size_t kEpiBytes = (size_t)4 * kEpiWarpFloats * sizeof(float);  // 4 epilogue warps

// `ybase`: the block's row 0, column 0 in Y; `ld`: Y's row stride in floats.
__device__ __forceinline__ void store_block_rows(float* tile, const uint32_t (&v)[32], float* ybase,
                                                 size_t ld, int rows_valid, int cols_valid, int lane) {
    float4* mine = reinterpret_cast<float4*>(tile + lane * kEpiStride);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        mine[k] = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                              __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
    __syncwarp();
    const int sub = lane >> 3;        // row within a group of 4
    const int col = (lane & 7) * 4;   // first of this lane's 4 columns
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int row = 4 * j + sub;
        if (row < rows_valid && col < cols_valid)
            __stcs(reinterpret_cast<float4*>(ybase + (size_t)row * ld + col),
                   *reinterpret_cast<const float4*>(tile + row * kEpiStride + col));
    }
    __syncwarp();
}

// Combine epilogue: the same transposed block, each row scaled by its slot's gate and
// written into its token's row of `out`: stored by the token's first contribution (its
// lowest expert), added with a 16-byte fp32 reduction (red.global.add) by the others,
// which run only once the lower contributions have landed (combine_wait_lower).  `col0`:
// Y column of the block's column 0; `c`: the combine row of the block's row `lane`.
struct CombineRow {
    int tok;    // token of the row (0 past the tile's rows)
    float w;    // gate of the row's slot
    int first;  // 1: the token's lowest expert (store), 0: a later one (add)
};

__device__ __forceinline__ void red_block_rows(float* tile, const uint32_t (&v)[32], float* out, size_t ld,
                                               int col0, int rows_valid, int cols_valid, int lane,
                                               const CombineRow& c) {
    float4* mine = reinterpret_cast<float4*>(tile + lane * kEpiStride);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        mine[k] = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                              __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
    __syncwarp();
    const int sub = lane >> 3;
    const int col = (lane & 7) * 4;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int row = 4 * j + sub;
        const int t = __shfl_sync(kFull, c.tok, row);
        const float w = __shfl_sync(kFull, c.w, row);
        const int first = __shfl_sync(kFull, c.first, row);
        if (row < rows_valid && col < cols_valid) {
            float4 y = *reinterpret_cast<const float4*>(tile + row * kEpiStride + col);
            y.x *= w;
            y.y *= w;
            y.z *= w;
            y.w *= w;
            float4* dst = reinterpret_cast<float4*>(out + (size_t)t * ld + col0 + col);
            if (first) *dst = y;
            else atomicAdd(dst, y);
        }
    }
    __syncwarp();
}

// Combine: token, gate and order of tile row `r` (this lane's row), or (0, 0, 1) past
// the tile's rows.  The row is its token's first contribution when no other slot of the
// token has a lower destination row (destination rows are expert-major, so that slot's
// expert would be lower).
__device__ __forceinline__ CombineRow combine_row(const DispatchGemmParams& p, int row0, int r, int rows) {
    CombineRow c{0, 0.f, 1};
    if (r < rows) {
        const int row = row0 + r;
        const int s = __ldg(p.perm + row);
        c.tok = s / p.k;
        c.w = __ldg(p.topk_w + s);
        for (int j = 0; j < p.k; ++j)
            if (__ldg(p.dest + c.tok * p.k + j) < row) c.first = 0;
    }
    return c;
}

// Combine completion word of column tile n of the 128-row tile `mtile`: word 0, or for an
// M=128 pair tile (whose two CTAs each hold 64 of its rows) word `half` of that CTA.
__device__ __forceinline__ uint32_t* combine_flag(const DispatchGemmParams& p, int mtile, int n, int half) {
    return p.cflags + ((size_t)mtile * p.n_tiles + n) * 2 + half;
}

// Waits (this lane) until every lower contribution of the token of tile row `r` to
// column tile n has landed: for each other slot of the token whose destination row r2
// is below this row, the completion word of r2's 128-row tile (or, for an M=128 pair
// tile, of r2's 64-row half) in column tile n holds the call's epoch.  Such tiles
// belong to lower experts and were claimed earlier, so the wait always ends; it is
// still bounded (MOE_ERR_TIMEOUT, then the row proceeds).
__device__ void combine_wait_lower(const DispatchGemmParams& p, const int* mt_base, bool pair, int row0, int r,
                                   int rows, int n, const CombineRow& c, const Waiter& w) {
    if (r >= rows || c.first) return;
    const int row = row0 + r;
    for (int j = 0; j < p.k; ++j) {
        const int r2 = __ldg(p.dest + c.tok * p.k + j);
        if (r2 >= row) continue;
        int lo = 0, hi = p.E;  // the expert holding r2: the largest e with offsets[e] <= r2
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(p.offsets + mid) <= r2) lo = mid;
            else hi = mid;
        }
        const int seg = __ldg(p.offsets + lo);
        const int lt = (r2 - seg) / kTileM;
        int half = 0;
        if (pair) {
            const int cnt = __ldg(p.offsets + lo + 1) - seg;
            if (cnt - 2 * kTileM * (lt >> 1) <= kTileM) half = (r2 - seg - kTileM * lt) >= kTileM / 2 ? 1 : 0;
        }
        const uint32_t* f = combine_flag(p, mt_base[lo] + lt, n, half);
        if (ld_acquire_gpu(f) == w.epoch) continue;
        const uint64_t t0 = global_timer_ns();
        for (uint32_t i = 1;; ++i) {
            if (ld_acquire_gpu(f) == w.epoch) break;
            if ((i & 31u) == 0 && global_timer_ns() - t0 > (uint64_t)w.flag_timeout_ns) {
                report_error(w.status, kStTimeout, -4, row, (int)w.epoch);
                break;
            }
        }
    }
}

// After a tile's combine stores: every epilogue thread fences its stores and reductions,
// the four epilogue warps meet at named barrier 1, and one thread releases the tile's
// completion word for column tile n with the call's epoch.
__device__ __forceinline__ void combine_publish(const DispatchGemmParams& p, int mtile, int n, int half,
                                               uint32_t epoch) {
    __threadfence();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (threadIdx.x == kEpiWarp0 * 32 && mtile >= 0) st_release_gpu(combine_flag(p, mtile, n, half), epoch);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x = lo: the lower address
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Gated (SwiGLU) activation: h = silu(g) * u with silu(g) = g / (1 + e^-g), fp32,
// rounded once to bf16 (nearest even).
__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Epilogue of one accumulator (single or pair tile, `bn` columns) for one warp's
// 32-row lane quarter: Y in fp32 or bf16, or in gated mode H = silu(gate) * up in
// bf16 from the gate columns [0, bn/2) and the up columns [bn/2, bn).  bf16 output
// goes 64 columns at a time, packed into 32 words per row, so that it leaves
// through the same full-line (128-byte) row stores as a 32-column fp32 block.
__device__ __forceinline__ void epilogue_tile(const DispatchGemmParams& p, const TileInfo& ti, int bn,
                                              uint32_t tbase, int q, int lane, float* epi,
                                              const CombineRow& cr) {
    const int rows_valid = min(32, ti.rows - 32 * q);  // rows of this warp's lane quarter
    // output columns of the tile (TMEM columns from 0): the whole tile or one half
    const int cw = ti.half ? bn / 2 : bn;
    const int c0 = ti.n * bn + (ti.half ? (ti.half - 1) * cw : 0);
    if (p.glu) {
        const int half = bn / 2;
        const int fcols = min(half, p.F - ti.n * half);
        uint16_t* hbase = p.H + (size_t)(ti.row0 + 32 * q) * p.F + (size_t)ti.n * half;
        for (int c = 0; c < fcols; c += 64) {
            uint32_t w[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t g[32], u[32];
                tmem_ld_32x32(tbase + (uint32_t)(c + 32 * h), g);
                tmem_ld_32x32(tbase + (uint32_t)(half + c + 32 * h), u);
                tmem_ld_wait(g);
                tmem_ld_wait(u);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[16 * h + i] = pack_bf16x2(swiglu(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                                                swiglu(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1])));
            }
            if (rows_valid > 0)
                store_block_rows(epi, w, reinterpret_cast<float*>(hbase + c), (size_t)p.F / 2, rows_valid,
                                 (fcols - c) / 2, lane);
        }
    } else if (p.out_bf16) {
        uint16_t* ybase = static_cast<uint16_t*>(p.Y) + (size_t)(ti.row0 + 32 * q) * p.N + (size_t)c0;
        const int ncols = min(cw, p.N - c0);
        for (int c = 0; c < ncols; c += 64) {
            uint32_t w[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t v[32];
                tmem_ld_32x32(tbase + (uint32_t)(c + 32 * h), v);
                tmem_ld_wait(v);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[16 * h + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            }
            if (rows_valid > 0)
                store_block_rows(epi, w, reinterpret_cast<float*>(ybase + c), (size_t)p.N / 2, rows_valid,
                                 (ncols - c) / 2, lane);
        }
    } else if (p.combine) {
        const int ncols = min(bn, p.N - ti.n * bn);
        for (int c = 0; c < ncols; c += 32) {
            uint32_t v[32];
            tmem_ld_32x32(tbase + (uint32_t)c, v);
            tmem_ld_wait(v);
            if (rows_valid > 0)
                red_block_rows(epi, v, p.out, (size_t)p.N, ti.n * bn + c, rows_valid, ncols - c, lane, cr);
        }
    } else {
        float* ybase = static_cast<float*>(p.Y) + (size_t)(ti.row0 + 32 * q) * p.N + (size_t)c0;
        const int ncols = min(cw, p.N - c0);
        for (int c = 0; c < ncols; c += 32) {
            uint32_t v[32];
            tmem_ld_32x32(tbase + (uint32_t)c, v);
            tmem_ld_wait(v);
            if (rows_valid > 0) store_block_rows(epi, v, ybase + c, (size_t)p.N, rows_valid, ncols - c, lane);
        }
    }
}

// Epilogue of an M=128 pair tile for this CTA's 64 rows.  Such an MMA leaves, for
// every 256-column MMA h of the tile, rows 0-63 of its columns [0, 128) in TMEM
// lanes 0-63 and of its columns [128, 256) in lanes 64-127, all in TMEM columns
// [256 h, 256 h + 128).  So lane quarter q holds rows 32 (q & 1) .. + 31 and
// tile columns 256 h + 128 (q >> 1) + [0, 128).  `tacc`: the accumulator's TMEM
// address.  Not used for gated tiles, whose gate and up columns would then lie
// in different warps.
__device__ __forceinline__ void epilogue_tile_m128(const DispatchGemmParams& p, const TileInfo& ti, int bn,
                                                   uint32_t tacc, int q, int lane, float* epi,
                                                   const CombineRow& cr) {
    const int rb = q & 1, ch = q >> 1;
    const int rows_valid = min(32, ti.rows - 32 * rb);
    if (rows_valid <= 0) return;  // warp-uniform
    const uint32_t tq = tacc + ((uint32_t)(32 * q) << 16);
    const size_t row = (size_t)(ti.row0 + 32 * rb);
    for (int h = 0; h < bn / 256; ++h) {
        const int col0 = ti.n * bn + 256 * h + 128 * ch;  // first Y column of this warp's block
        const int ncols = min(128, p.N - col0);
        if (ncols <= 0) continue;
        const uint32_t t0 = tq + (uint32_t)(256 * h);
        if (p.out_bf16) {
            uint16_t* ybase = static_cast<uint16_t*>(p.Y) + row * p.N + col0;
            for (int c = 0; c < ncols; c += 64) {
                uint32_t w[32];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t v[32];
                    tmem_ld_32x32(t0 + (uint32_t)(c + 32 * hh), v);
                    tmem_ld_wait(v);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[16 * hh + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                }
                store_block_rows(epi, w, reinterpret_cast<float*>(ybase + c), (size_t)p.N / 2, rows_valid,
                                 (ncols - c) / 2, lane);
            }
        } else if (p.combine) {
            for (int c = 0; c < ncols; c += 32) {
                uint32_t v[32];
                tmem_ld_32x32(t0 + (uint32_t)c, v);
                tmem_ld_wait(v);
                red_block_rows(epi, v, p.out, (size_t)p.N, col0 + c, rows_valid, ncols - c, lane, cr);
            }
        } else {
            float* ybase = static_cast<float*>(p.Y) + row * p.N + col0;
            for (int c = 0; c < ncols; c += 32) {
                uint32_t v[32];
                tmem_ld_32x32(t0 + (uint32_t)c, v);
                tmem_ld_wait(v);
                store_block_rows(epi, v, ybase + c, (size_t)p.N, rows_valid, ncols - c, lane);
            }
        }
    }
}

// First column in W of the 64-column B box `j` of a tile whose columns start at
// `ncol` (plain) or, in gated mode, whose gate and up halves each hold `half`
// columns starting at F-column n * half: boxes [0, half/64) are gate columns,
// the rest the matching up columns F + ...
__device__ __forceinline__ int b_box_col(const DispatchGemmParams& p, int n, int bn, int j) {
    if (!p.glu) return n * bn + 64 * j;
    const int half = bn / 2;
    const int hb = half / 64;
    const int up = j >= hb ? 1 : 0;
    return up * p.F + n * half + 64 * (j - up * hb);
}

template <int BN, int STAGES>
struct Cfg {
    static constexpr int kABytes = kTileM * kTileK * 2;  // 16 KB
    static constexpr int kBBytes = BN * kTileK * 2;      // BN/64 boxes of 64 x 64
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kIdesc = idesc_bf16_f32_kmajA_mnmajB(kTileM, BN);
    static constexpr uint32_t kIdescHalf = idesc_bf16_f32_kmajA_mnmajB(kTileM, BN / 2);  // split tiles
    static constexpr int kTmemCols = 2 * BN <= 256 ? 256 : 512;  // allocations are powers of two
    static constexpr size_t kSmem =
        1024 + (size_t)STAGES * kStageBytes + kEpiBytes + sizeof(SmemCtl) + 2 * sizeof(int) * (kMaxE + 1);
    static_assert(STAGES <= kMaxStages, "stages");
    static_assert(kSmem <= 232448, "more than 227 KB of shared memory per CTA");
    static_assert(BN == 128 || BN == 192 || BN == 256, "tile_n");
    // the scatter stages rows in the stage area: 8 warps x 32 lanes x slots x 16 B
    static constexpr int kScatterSlots = scatter_slots_per_lane((size_t)STAGES * kStageBytes);
    static_assert(kScatterSlots >= 32, "stage area too small for the scatter staging (two pieces per warp)");
    static_assert((size_t)kScatterSlots * 16 * 32 * (kThreads / 32) <= (size_t)STAGES * kStageBytes,
                  "scatter staging must stay inside the stage area");
};

// The TMA thread claims the next tile, publishes its description to the MMA and
// epilogue warps and reads its ready flag a few k-blocks before it has issued
// the current tile, so the claim and flag latencies overlap the loads still
// buffered ahead of the MMA.
constexpr int kLookaheadKb = 4;
// CTA pairs claim earlier, at k-block kPairClaimKb of the current tile: their TMA
// thread is busy issuing for most of a tile, and a claim at the end of a short tile
// (d = 2048: 32 k-blocks) stalls its issue while the ring is least full.
constexpr int kPairClaimKb = 2;

template <int BN, int STAGES>
__device__ void tma_role(const DispatchGemmParams& p, SmemCtl* ctl, const int* mt_base,
                         uint8_t* sA, uint8_t* sB, const Waiter& w) {
    using C = Cfg<BN, STAGES>;
    const uint32_t total_tiles = (uint32_t)mt_base[p.E] * (uint32_t)p.n_tiles;
    // claims below split_from are whole tiles; each tile from split_from on is claimed twice,
    // as its left and its right half.  split_from is 0 (every tile split) when the schedule
    // fills at most half the grid (half_tiles 1) or always (half_tiles 2), else total_tiles.
    const bool split = p.half_tiles == 2 || (p.half_tiles == 1 && 2u * total_tiles <= gridDim.x);
    const uint32_t split_from = split ? 0u : total_tiles;
    const uint32_t total_claims = 2u * total_tiles - split_from;
    // a schedule of 2-8 waves of claims: only as many CTAs claim as fill every wave (the
    // others leave after their scatter share), so that an HBM-bound layer's CTAs end
    // together instead of a partial last wave running on a few of them
    bool claims = true;
    {
        const uint32_t g = gridDim.x;
        const uint32_t waves = (total_claims + g - 1) / g;
        if (waves >= 2 && waves <= 8) claims = (uint32_t)ctl->role < (total_claims + waves - 1) / waves;
    }
    const int e_per_rank = p.E / p.R;
    tma_prefetch_map(&p.b_map);
    if (!p.gather)  // no A tensor map in the gather mode
        for (int r = 0; r < p.R; ++r) tma_prefetch_map(&p.a_map[r]);
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;
    uint32_t sphase = 0;
    int last_phase[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) last_phase[s] = -1;

    // claim a tile, describe it, hand it to the MMA and epilogue warps, read its flag
    auto push_next = [&](TileInfo& ti, uint32_t& flag) -> bool {
        if (!wait_bar(smem_addr(&ctl->sempty[slot]), sphase ^ 1u, w, 1)) return false;
        const uint32_t claim = claims ? atomicAdd(p.hdr + kHdrTileCtr, 1u) : total_claims;
        if (claim >= total_claims) {
            ti.e = ti.m = ti.n = ti.mtile = ti.row0 = ti.rank = ti.arow = ti.m128 = ti.half = 0;
            ti.rows = -1;
        } else {
            const uint32_t tile = claim < split_from ? claim : split_from + (claim - split_from) / 2;
            ti.half = claim < split_from ? 0 : 1 + (int)((claim - split_from) & 1u);
            const int u = (int)(tile / (uint32_t)p.n_tiles);
            const int e = expert_of(mt_base, p.E, u);
            const int mt_e = mt_base[e + 1] - mt_base[e];
            const int local = (int)(tile - (uint32_t)mt_base[e] * (uint32_t)p.n_tiles);
            // bands of `band` row tiles (the last may be shorter); inside a band the
            // column tile is the slow index, so a band's rows are needed first and
            // each weight panel is reused by the band's row tiles while hot in L2
            const int bh = p.band > 0 ? p.band : mt_e;
            const int b = local / (bh * p.n_tiles);
            const int rem = local - b * bh * p.n_tiles;
            const int h = min(bh, mt_e - b * bh);
            ti.e = e;
            ti.n = rem / h;
            ti.m = b * bh + rem % h;
            ti.mtile = mt_base[e] + ti.m;
            const int seg0 = __ldg(p.offsets + e);
            const int cnt = __ldg(p.offsets + e + 1) - seg0;
            ti.row0 = seg0 + ti.m * kTileM;
            ti.rows = min(kTileM, cnt - ti.m * kTileM);
            ti.rank = e / e_per_rank;
            ti.arow = ti.row0 - __ldg(p.offsets + ti.rank * e_per_rank);
            ti.m128 = 0;
        }
        ctl->ring[slot] = ti;
        mbar_arrive(smem_addr(&ctl->sfull[slot]));
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        flag = (ti.rows > 0 && !p.a_ready && !p.gather) ? ld_acquire_gpu(p.flags + ti.mtile) : w.epoch;
        return true;
    };

    TileInfo cur;
    uint32_t cur_flag = 0;
    bool ok = push_next(cur, cur_flag);
    bool first = true;
    while (ok && cur.rows >= 0) {
        if (p.trace) {
            const unsigned long long t0 = global_timer_ns();
            if (cur_flag != w.epoch) wait_flag(p.flags + cur.mtile, w, cur.mtile, cur.e);
            const unsigned long long t1 = global_timer_ns();
            trace_add(p, kTrFlagWait, t1 - t0);
            trace_add(p, kTrTiles, 1);
            if (first) trace_set(p, kTrFirstTile, t1);
            first = false;
        } else if (cur_flag != w.epoch) {
            wait_flag(p.flags + cur.mtile, w, cur.mtile, cur.e);
        }
        fence_proxy_async_global();
        const CUtensorMap* amap = &p.a_map[cur.rank];
        const int brow = cur.e * p.d;
        // B boxes of the tile: all BN/64, or the BN/128 of one half (split tiles are never
        // gated, so a half's boxes are consecutive columns)
        const int nbox = cur.half ? BN / 128 : BN / 64;
        const int bshift = cur.half == 2 ? BN / 2 : 0;
        const uint32_t b_bytes = (uint32_t)nbox * 8192u;
        const int pre_kb = p.k_blocks > kLookaheadKb ? p.k_blocks - kLookaheadKb : 0;
        TileInfo nxt;
        uint32_t nxt_flag = 0;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (kb == pre_kb && !push_next(nxt, nxt_flag)) {
                ok = false;
                break;
            }
            if (!wait_bar(smem_addr(&ctl->empty[stage]), phase ^ 1u, w, 2)) {
                ok = false;
                break;
            }
            const uint32_t fb = smem_addr(&ctl->full[stage]);
            if (p.gather) {  // the gather warps fill A and arrive on the same barrier
                mbar_arrive_expect_tx(fb, b_bytes);
            } else {
                mbar_arrive_expect_tx(fb, C::kABytes + b_bytes);
                tma_load_2d(smem_addr(sA + stage * C::kABytes), amap, fb, kb * kTileK, cur.arow);
            }
            if (p.gather) {  // otherwise warp 2 issues the B boxes (tma_b_role)
#pragma unroll
                for (int j = 0; j < BN / 64; ++j)
                    if (j < nbox)
                        tma_load_2d(smem_addr(sB + stage * C::kBBytes + j * 8192), &p.b_map, fb,
                                    b_box_col(p, cur.n, BN, j) + bshift, brow + kb * kTileK);
            }
            last_phase[stage] = (int)phase;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        cur = nxt;
        cur_flag = nxt_flag;
    }
    if (p.trace) trace_set(p, kTrIssueEnd, global_timer_ns());
    // no TMA write may still be landing in shared memory when the CTA exits
#pragma unroll
    for (int s = 0; s < STAGES; ++s)
        if (last_phase[s] >= 0) wait_bar(smem_addr(&ctl->full[s]), (uint32_t)last_phase[s], w, 3, false);
}

// B loads of a single-CTA tile outside the gather mode (lane 0 of warp 2): follows the
// schedule ring and issues the tile's B boxes (or one half's) of every k-block once the
// stage is free; the TMA thread issues A and arms the stage for all its bytes.
template <int BN, int STAGES>
__device__ void tma_b_role(const DispatchGemmParams& p, SmemCtl* ctl, uint8_t* sB, const Waiter& w) {
    using C = Cfg<BN, STAGES>;
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;
    uint32_t sphase = 0;
    for (;;) {
        if (!wait_bar(smem_addr(&ctl->sfull[slot]), sphase, w, 35)) return;
        const TileInfo ti = ctl->ring[slot];
        mbar_arrive(smem_addr(&ctl->sempty[slot]));
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        if (ti.rows < 0) return;
        const int nbox = ti.half ? BN / 128 : BN / 64;
        const int bshift = ti.half == 2 ? BN / 2 : 0;
        const int brow = ti.e * p.d;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!wait_bar(smem_addr(&ctl->empty[stage]), phase ^ 1u, w, 36)) return;
            const uint32_t fb = smem_addr(&ctl->full[stage]);
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
                if (j < nbox)
                    tma_load_2d(smem_addr(sB + stage * C::kBBytes + j * 8192), &p.b_map, fb,
                                b_box_col(p, ti.n, BN, j) + bshift, brow + kb * kTileK);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

template <int BN, int STAGES, bool GATHER>
__device__ void mma_role(const DispatchGemmParams& p, SmemCtl* ctl, uint8_t* sA, uint8_t* sB,
                         uint32_t tmem_base, const Waiter& w) {
    using C = Cfg<BN, STAGES>;
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;
    uint32_t sphase = 0;
    int acc = 0;
    uint32_t aphase = 0;
    bool ok = true;
    while (ok) {
        if (!wait_bar(smem_addr(&ctl->sfull[slot]), sphase, w, 4)) break;
        const int rows = ctl->ring[slot].rows;
        const uint32_t idesc = ctl->ring[slot].half ? C::kIdescHalf : C::kIdesc;  // N = BN or BN/2
        mbar_arrive(smem_addr(&ctl->sempty[slot]));
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        if (rows < 0) break;
        if (!wait_bar(smem_addr(&ctl->tempty[acc]), aphase ^ 1u, w, 5)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        // k-blocks of four K=16 steps in the loop; a last k-block of a reduction that is
        // not a multiple of 64 (fewer steps: the loaded columns past d, zero-filled A and the
        // next expert's W rows, are not used) after it, so that the loop body stays lean:
        // the MMA thread's issue latency is on the critical path
        const int kfull = p.last_ksteps == kTileK / kUmmaK ? p.k_blocks : p.k_blocks - 1;
        for (int kb = 0; kb < kfull; ++kb) {
            if (!wait_bar(smem_addr(&ctl->full[stage]), phase, w, 6)) {
                ok = false;
                break;
            }
            if (GATHER) fence_proxy_async_smem();  // the gather threads' rows
            tc_fence_after();
            const uint32_t a0 = smem_addr(sA + stage * C::kABytes);
            const uint32_t b0 = smem_addr(sB + stage * C::kBBytes);
#pragma unroll
            for (int kk = 0; kk < kTileK / kUmmaK; ++kk) {
                // A: K-major rows of 128 B, 8-row groups 1024 B apart; K step = +32 B.
                // B: N-major, 64-column boxes 8 KB apart (LBO), 8-row K groups
                //    1024 B apart (SBO); K step of 16 rows = +2048 B.
                const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
                const uint64_t bd = smem_desc_sw128(b0 + kk * 2048, 8192, 1024);
                umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            umma_commit(smem_addr(&ctl->empty[stage]));
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (ok && kfull < p.k_blocks) {  // the short last k-block
            if (!wait_bar(smem_addr(&ctl->full[stage]), phase, w, 6)) break;
            if (GATHER) fence_proxy_async_smem();
            tc_fence_after();
            const uint32_t a0 = smem_addr(sA + stage * C::kABytes);
            const uint32_t b0 = smem_addr(sB + stage * C::kBBytes);
            for (int kk = 0; kk < p.last_ksteps; ++kk) {
                const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
                const uint64_t bd = smem_desc_sw128(b0 + kk * 2048, 8192, 1024);
                umma_bf16(d_tmem, ad, bd, idesc, (kfull | kk) != 0 ? 1u : 0u);
            }
            umma_commit(smem_addr(&ctl->empty[stage]));
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        umma_commit(smem_addr(&ctl->tfull[acc]));
        acc ^= 1;
        if (acc == 0) aphase ^= 1u;
    }
    // every MMA issued by this thread completes before TMEM is released
    umma_commit(smem_addr(&ctl->mma_done));
    wait_bar(smem_addr(&ctl->mma_done), 0u, w, 7, false);
}

template <int BN, int STAGES>
__device__ void epilogue_role(const DispatchGemmParams& p, SmemCtl* ctl, uint32_t tmem_base,
                              const Waiter& w, float* epi, const int* mt_base) {
    const int lane = threadIdx.x & 31;
    const int q = (threadIdx.x >> 5) & 3;  // TMEM lane quarter of this warp
    int slot = 0;
    uint32_t sphase = 0;
    int acc = 0;
    uint32_t aphase = 0;
    for (;;) {
        const bool got = wait_bar(smem_addr(&ctl->sfull[slot]), sphase, w, 8);
        if (!__all_sync(kFull, got)) break;
        const TileInfo ti = ctl->ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl->sempty[slot]));
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        if (ti.rows < 0) break;
        const bool ready = wait_bar(smem_addr(&ctl->tfull[acc]), aphase, w, 9);
        if (!__all_sync(kFull, ready)) break;
        tc_fence_after();
        CombineRow cr{0, 0.f, 1};
        if (p.combine) {
            cr = combine_row(p, ti.row0, 32 * q + lane, ti.rows);
            combine_wait_lower(p, mt_base, false, ti.row0, 32 * q + lane, ti.rows, ti.n, cr, w);
            __syncwarp();
        }
        const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(32 * q) << 16);
        epilogue_tile(p, ti, BN, tbase, q, lane, epi, cr);
        tc_fence_before();
        mbar_arrive(smem_addr(&ctl->tempty[acc]));
        if (p.combine) combine_publish(p, ti.mtile, ti.n, 0, w.epoch);
        acc ^= 1;
        if (acc == 0) aphase ^= 1u;
    }
}

// Direct-gather A loads (gather mode, warps 2 and 3 of every CTA): for every tile
// the warps take from the schedule ring, warp `part` copies the CTA's rows
// [64 part, 64 part + 64) of the tile straight from their token rows of x
// (perm[row] / k) into the stage's A buffer with 16-byte cp.async, in the
// 128-byte-swizzled K-major layout the MMA descriptors expect (16-byte chunk c of
// row r lands at r*128 + (c ^ (r%8))*16).  Eight lanes cover one row's 128 bytes of
// a k-block, so each copy instruction moves four whole 128-byte lines.  Rows past
// the tile's valid rows are zero-filled.  Every thread ends a stage's copies with a
// cp.async-completion arrival (.noinc) on the stage's barrier, so a stage is
// published as soon as its rows have landed and the warps never wait for their own
// copies: on the full barrier (with the B bytes) in single CTAs and the pair leader,
// on the CTA's own `afull` barrier in the pair peer, whose relay thread
// (pair_relay_role) passes each completed stage on to the leader.  The consumers
// fence the copies for the async proxy (the tensor cores read shared memory there)
// after their wait: the MMA thread for its CTA's rows, the relay for the peer's.  No
// receive buffer is written and no ready flag is read.  The copies are cp.async by
// warps, not TMA: a TMA gather of four 128-byte rows (tile::gather4) per lane ran
// about 3x slower than this here (32 small TMA operations per k-block and CTA).
constexpr int kGatherWarp0 = 2;
constexpr int kGatherWarps = 2;
constexpr int kGatherRows = kTileM / kGatherWarps;  // rows per warp
template <int STAGES>
__device__ void gather_a_role(const DispatchGemmParams& p, SmemCtl* ctl, uint8_t* sA, const Waiter& w,
                              int part, bool pair, bool leader, uint32_t lead) {
    constexpr int kABytes = kTileM * kTileK * 2;  // 128 rows x 64 columns
    constexpr int kIters = kGatherRows / 4;
    const int lane = threadIdx.x & 31;
    const char* xb = reinterpret_cast<const char*>(p.x);
    const size_t row_bytes = (size_t)p.d * 2;
    int slot = 0;
    uint32_t sphase = 0;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    while (ok) {
        const bool got = wait_bar(smem_addr(&ctl->sfull[slot]), sphase, w, 40, true, pair);
        if (!__all_sync(kFull, got)) break;
        const TileInfo ti = ctl->ring[slot];
        __syncwarp();
        if (lane == 0) {
            const uint32_t se = smem_addr(&ctl->sempty[slot]);
            if (leader) mbar_arrive(se);
            else mbar_arrive_remote(mapa_shared(se, lead));
        }
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        if (pair ? ti.e < 0 : ti.rows < 0) break;
        // this lane copies chunk c of the warp's rows 4i + lane/8 (i < 16): their
        // token rows, gathered from the lanes that read perm, stay in registers
        const int c = lane & 7;
        const int r0 = part * kGatherRows;
        int tok[kIters];  // -1: past the tile's valid rows
        {
            int mine[kGatherRows / 32];
#pragma unroll
            for (int j = 0; j < kGatherRows / 32; ++j) {
                const int r = r0 + lane + 32 * j;
                mine[j] = r < ti.rows ? __ldg(p.perm + ti.row0 + r) / p.k : -1;
            }
#pragma unroll
            for (int i = 0; i < kIters; ++i) {
                // warp row 4i + lane/8 is held by lane (4i + lane/8) % 32 in mine[i / 8]
                const int src_lane = (4 * i + (lane >> 3)) & 31;
                tok[i] = __shfl_sync(kFull, mine[i / 8], src_lane);
            }
        }
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            bool free_ok = true;
            if (lane == 0) free_ok = wait_bar(smem_addr(&ctl->empty[stage]), phase ^ 1u, w, 41, true, pair);
            if (!__shfl_sync(kFull, free_ok ? 1 : 0, 0)) {
                ok = false;
                break;
            }
            const uint32_t a0 = smem_addr(sA + stage * kABytes);
            // this lane's 8 columns start at kb * 64 + 8 c; past d (a last k-block of a
            // reduction that is not a multiple of 64) nothing is read and zeros are written
            const bool in_row = kb * kTileK + 8 * c < p.d;
            const size_t kofs = in_row ? (size_t)kb * (kTileK * 2) + 16 * c : 0;
#pragma unroll
            for (int i = 0; i < kIters; ++i) {
                const int r = r0 + 4 * i + (lane >> 3);
                const int t = tok[i];
                cp_async16_cg_zfill(a0 + (uint32_t)r * 128u + (uint32_t)((c ^ (r & 7)) << 4),
                                    xb + (size_t)(t < 0 ? 0 : t) * row_bytes + kofs, (t < 0 || !in_row) ? 0 : 16);
            }
            cp_async_mbar_arrive_noinc(smem_addr(leader ? &ctl->full[stage] : &ctl->afull[stage]));
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    // no copy may still be landing when the CTA leaves (also after an abort)
    cp_async_wait_all();
}

// Gather mode, peer CTA of a pair (its otherwise idle warp 1, lane 0): follows the
// schedule ring and, for every stage, waits until the peer's gather warps have landed
// their A rows (the peer's `afull` barrier) and then arrives on the leader's stage
// barrier, which the leader's MMA thread waits on.  One remote arrival per stage
// from this thread, instead of one from each gather thread.
template <int STAGES>
__device__ void pair_relay_role(const DispatchGemmParams& p, SmemCtl* ctl, const Waiter& w, uint32_t lead) {
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;
    uint32_t sphase = 0;
    for (;;) {
        if (!wait_bar(smem_addr(&ctl->sfull[slot]), sphase, w, 31, true, true)) return;
        const int e = ctl->ring[slot].e;
        mbar_arrive_remote(mapa_shared(smem_addr(&ctl->sempty[slot]), lead));
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        if (e < 0) return;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            // afull's arrivals are this CTA's own copies: a CTA-scope wait
            if (!wait_bar(smem_addr(&ctl->afull[stage]), phase, w, 32, true, false)) return;
            fence_proxy_async_smem();  // the gathered rows, before the leader's MMAs read them
            mbar_arrive_remote(mapa_shared(smem_addr(&ctl->full[stage]), lead));
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    dispatch_gemm_kernel(const __grid_constant__ DispatchGemmParams p) {
    using C = Cfg<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * C::kABytes;
    float* epi_tiles = reinterpret_cast<float*>(sB + STAGES * C::kBBytes);  // 4 x 32 x 36 fp32
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(reinterpret_cast<uint8_t*>(epi_tiles) + kEpiBytes);
    int* mt_base = reinterpret_cast<int*>(ctl + 1);  // row tiles per expert, prefix
    int* unit_base = mt_base + (kMaxE + 1);           // scatter units per expert, prefix

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), p.gather ? 1 + 32 * kGatherWarps : 1);  // + gather threads
            mbar_init(smem_addr(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_addr(&ctl->tfull[a]), 1);
            mbar_init(smem_addr(&ctl->tempty[a]), 128);
        }
        for (int r = 0; r < kRing; ++r) {
            mbar_init(smem_addr(&ctl->sfull[r]), 1);
            // MMA thread + 4 epilogue warps (+ the gather warps)
            mbar_init(smem_addr(&ctl->sempty[r]), 1 + 4 + (p.gather ? kGatherWarps : 1));
        }
        mbar_init(smem_addr(&ctl->mma_done), 1);
        ctl->abort = 0;
        ctl->role = (int)atomicAdd(p.hdr + kHdrRoleCtr, 1u);
        uint32_t ep = __ldcg(p.hdr + kHdrEpoch) + 1u;
        ctl->epoch = ep == 0u ? 1u : ep;
        mbar_fence_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_addr(&ctl->tmem_base), C::kTmemCols);
        tmem_relinquish();
    }
    build_expert_table(p.offsets, p.E, kTileM, mt_base, ctl->wsum);  // contain __syncthreads
    build_expert_table(p.offsets, p.E, kRowsPerChunk, unit_base, ctl->wsum, p.nch);
    if (mt_base[p.E] > p.max_mtiles || __ldg(p.offsets + p.E) != p.T * p.k) {
        // offsets that do not describe T*k rows: report, and schedule nothing
        __syncthreads();
        if (tid == 0) {
            report_error(p.status, kStDevice, -2, __ldg(p.offsets + p.E), 0);
            for (int e = 0; e <= p.E; ++e) mt_base[e] = 0;
            for (int i = 0; i <= p.nch * p.E; ++i) unit_base[i] = 0;
        }
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const uint32_t epoch = ctl->epoch;
    const int role = ctl->role;
    if (tid == 0 && p.trace) {  // the same thread runs the TMA role: no other writer yet
        for (int i = 0; i < kTraceWords; ++i) trace_set(p, i, 0ull);
        trace_set(p, kTrStart, global_timer_ns());
        trace_set(p, kTrRole, (unsigned long long)role);
    }

    const long long pipe_timeout = p.timeout_ns * 2 > 500000000LL ? p.timeout_ns * 2 : 500000000LL;
    const Waiter w{&ctl->abort, p.status, p.timeout_ns, pipe_timeout, epoch};
    if (role < p.producer_ctas) {
        unsigned long long* w64 = reinterpret_cast<unsigned long long*>(p.hdr);
        if (tid == 0) atomicMax(w64 + kHdrScatterInvStart / 2, ~(unsigned long long)global_timer_ns());
        scatter_role(p, mt_base, unit_base, role, epoch, sA, ctl, C::kScatterSlots, unit_base[p.nch * p.E]);
        __syncthreads();
        if (tid == 0) {
            const unsigned long long t = global_timer_ns();
            atomicMax(w64 + kHdrScatterEnd / 2, t);
            trace_set(p, kTrScatterEnd, t);
        }
    }

    if (warp == 0) {
        if (lane == 0) tma_role<BN, STAGES>(p, ctl, mt_base, sA, sB, w);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            if (p.gather) mma_role<BN, STAGES, true>(p, ctl, sA, sB, tmem_base, w);
            else mma_role<BN, STAGES, false>(p, ctl, sA, sB, tmem_base, w);
        }
        __syncwarp();
    } else if (p.gather && warp >= kGatherWarp0 && warp < kGatherWarp0 + kGatherWarps) {
        gather_a_role<STAGES>(p, ctl, sA, w, warp - kGatherWarp0, false, true, 0);
    } else if (!p.gather && warp == 2) {
        if (lane == 0) tma_b_role<BN, STAGES>(p, ctl, sB, w);
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        epilogue_role<BN, STAGES>(p, ctl, tmem_base, w, epi_tiles + (warp - kEpiWarp0) * kEpiWarpFloats, mt_base);
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 0 && p.trace) trace_set(p, kTrEnd, global_timer_ns());
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(p.hdr + kHdrDoneCtr, 1u);
        if (prev == gridDim.x - 1) {  // every CTA has finished with the counters
            __threadfence();
            p.hdr[kHdrTileCtr] = 0u;
            p.hdr[kHdrRoleCtr] = 0u;
            p.hdr[kHdrDoneCtr] = 0u;
            p.hdr[kHdrEpoch] = epoch;
            // scatter window of this call, for measurement; accumulators back to zero
            unsigned long long* w64 = reinterpret_cast<unsigned long long*>(p.hdr);
            const unsigned long long inv = atomicExch(w64 + kHdrScatterInvStart / 2, 0ull);
            const unsigned long long end = atomicExch(w64 + kHdrScatterEnd / 2, 0ull);
            w64[kHdrLastScatterStart / 2] = ~inv;
            w64[kHdrLastScatterEnd / 2] = end;
            __threadfence();
        }
    }
}

// ------------------------------------------------------------------ CTA-pair mode
//
// For layers with many rows per expert, CTAs run in clusters of two and every
// GEMM tile is 256 rows x 256 columns, computed by tcgen05.mma.cta_group::2:
// the even CTA of the pair (the leader) issues the MMAs, each CTA holds 128
// rows of A and 128 of the 256 columns of B in its own shared memory, and each
// CTA's TMEM receives its 128 rows of the accumulator.  Per SM this halves the
// B operand traffic (TMA writes into shared memory and MMA reads from it).
// With BN = 512 (an opt-in tile width) a tile is 256 x 512: each K step issues
// two N=256 MMAs into TMEM columns 0-255 and 256-511, each CTA holds 256 of the
// 512 B columns, and the one 512-column accumulator fills TMEM (no overlap of a
// tile's epilogue with the next tile's MMAs).
//  * The leader claims tiles and writes each tile's description into both
//    CTAs' schedule rings (the peer's through distributed shared memory).
//  * Both CTAs' TMA loads complete on the leader's stage barrier; the
//    leader's MMA commit is multicast to both CTAs' stage-empty and
//    accumulator-full barriers; both CTAs' epilogues release the accumulator
//    on the leader's barrier.
//  * Each CTA waits for the ready flag of its own 128-row half.
//  * An expert's last tile of at most 128 rows runs as an M=128 pair MMA, 64
//    rows per CTA, both CTAs waiting for that one row tile's flag
//    (pair_half_info, epilogue_tile_m128).
// The scatter role is unchanged; a pair takes one role ticket and its two
// CTAs become scatter CTAs 2t and 2t+1.
template <int STAGES, int BN>
struct PairCfg {
    static_assert(BN == 256 || BN == 512, "pair tile widths: 256 or 512 columns");
    static constexpr int kABytes = kTileM * kTileK * 2;  // 16 KB: this CTA's 128 rows
    static constexpr int kBN = BN;                       // tile width of the pair
    static constexpr int kHalves = BN / 256;             // N=256 MMAs per K step
    static constexpr int kBBytes = (BN / 2) * kTileK * 2;  // this CTA's BN/2 columns: 16 or 32 KB
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kIdesc = idesc_bf16_f32_kmajA_mnmajB(2 * kTileM, 256);
    static constexpr uint32_t kIdesc128 = idesc_bf16_f32_kmajA_mnmajB(kTileM, 256);  // tail tiles
    static constexpr int kTmemCols = 512;                // two 256-column accumulators or one of 512
    static constexpr int kAccs = 512 / BN;               // accumulators (TMEM double buffer for 256)
    static constexpr size_t kSmem =
        1024 + (size_t)STAGES * kStageBytes + kEpiBytes + sizeof(SmemCtl) + 3 * sizeof(int) * (kMaxE + 1);
    static_assert(STAGES <= kMaxStages, "stages");
    static_assert(kSmem <= 232448, "more than 227 KB of shared memory per CTA");
    static constexpr int kScatterSlots = scatter_slots_per_lane((size_t)STAGES * kStageBytes);
    static_assert(kScatterSlots >= 32, "stage area too small for the scatter staging (two pieces per warp)");
    static_assert((size_t)kScatterSlots * 16 * 32 * (kThreads / 32) <= (size_t)STAGES * kStageBytes,
                  "scatter staging must stay inside the stage area");
};

// Tile description of one CTA's half of a pair tile.  An expert's last pair tile
// with at most 128 rows runs as an M=128 pair MMA (not in gated mode): each CTA
// holds 64 of its rows (rows [64 half, 64 half + 64) of the 128-row tile 2 m2),
// and both halves wait for that row tile's flag.  Each CTA still loads a whole
// 128-row A box (the rank buffer's one tensor map): the box's rows 64-127 lie
// past this CTA's 64 rows (the peer's rows, the next expert's rows that the
// scatter may still be writing, or rows past the buffer, zero-filled).  The
// M=128 MMA reads only rows 0-63 of each CTA's A tile, so those extra rows are
// never used and a race on them cannot change a result.
__device__ void pair_half_info(const DispatchGemmParams& p, const int* mt_base, int e, int m2,
                               int n, int half, TileInfo& ti) {
    const int e_per_rank = p.E / p.R;
    const int seg0 = __ldg(p.offsets + e);
    const int cnt = __ldg(p.offsets + e + 1) - seg0;
    ti.e = e;
    ti.n = n;
    ti.half = 0;
    ti.m128 = (!p.glu && cnt - 2 * kTileM * m2 <= kTileM) ? 1 : 0;
    if (ti.m128) {
        ti.m = 2 * m2;
        ti.row0 = seg0 + ti.m * kTileM + (kTileM / 2) * half;
        ti.rows = min(kTileM / 2, cnt - ti.m * kTileM - (kTileM / 2) * half);  // may be <= 0 for the odd half
        ti.mtile = mt_base[e] + ti.m;
    } else {
        const int m = 2 * m2 + half;  // 128-row tile of this half
        ti.m = m;
        ti.row0 = seg0 + m * kTileM;
        ti.rows = min(kTileM, cnt - m * kTileM);  // may be <= 0 for the odd half
        ti.mtile = ti.rows > 0 ? mt_base[e] + m : -1;
    }
    ti.rank = e / e_per_rank;
    ti.arow = ti.row0 - __ldg(p.offsets + ti.rank * e_per_rank);
}

template <int STAGES, int BN, bool GATHER>
__device__ void pair_tma_role(const DispatchGemmParams& p, SmemCtl* ctl, const int* mt_base,
                              const int* pt_base, uint8_t* sA, uint8_t* sB, const Waiter& w,
                              bool leader, uint32_t peer) {
    using C = PairCfg<STAGES, BN>;
    const uint32_t total_tiles = (uint32_t)pt_base[p.E] * (uint32_t)p.n_tiles;
    tma_prefetch_map(&p.b_map);
    if (p.b3d) tma_prefetch_map(&p.b3_map);
    if (!GATHER)  // no A tensor map in the gather mode
        for (int r = 0; r < p.R; ++r) tma_prefetch_map(&p.a_map[r]);
    const uint32_t lead = leader ? cluster_ctarank() : peer;  // rank of the leader CTA
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;
    uint32_t sphase = 0;
    int last_phase[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) last_phase[s] = -1;

    // Leader: claim a pair tile and publish both halves' descriptions (the peer's by
    // asynchronous stores into its ring slot that complete its ring barrier).  Peer:
    // take the next description from its ring; with `block` false it only takes one that
    // is already there.  Both read the ready flag of their own half.
    bool armed = false;  // peer: this use of the ring slot is armed
    auto next_tile = [&](TileInfo& ti, uint32_t& flag, bool block, bool& got) -> bool {
        got = false;
        if (leader) {
            if (!wait_bar(smem_addr(&ctl->sempty[slot]), sphase ^ 1u, w, 21, true, true)) return false;
            const uint32_t tile = atomicAdd(p.hdr + kHdrTileCtr, 1u);
            TileInfo other;
            if (tile >= total_tiles) {
                ti.e = ti.m = ti.n = ti.mtile = ti.row0 = ti.rows = ti.rank = ti.arow = ti.m128 = ti.half = 0;
                ti.e = -1;
                other = ti;
            } else {
                const int u = (int)(tile / (uint32_t)p.n_tiles);
                const int e = expert_of(pt_base, p.E, u);
                const int pt_e = pt_base[e + 1] - pt_base[e];
                const int local = (int)(tile - (uint32_t)pt_base[e] * (uint32_t)p.n_tiles);
                const int n = local / pt_e;
                const int m2 = local % pt_e;
                pair_half_info(p, mt_base, e, m2, n, 0, ti);
                pair_half_info(p, mt_base, e, m2, n, 1, other);
            }
            ctl->ring[slot] = ti;
            // the peer's half: asynchronous stores whose bytes complete the peer's ring
            // barrier (armed by the peer's TMA thread), so the description is visible there
            // when the barrier completes, without a cluster-scope release
            const int* o = reinterpret_cast<const int*>(&other);
            const uint32_t remote = mapa_shared(smem_addr(&ctl->ring[slot]), peer);
            const uint32_t rbar = mapa_shared(smem_addr(&ctl->sfull[slot]), peer);
#pragma unroll
            for (int i = 0; i < (int)(sizeof(TileInfo) / 8); ++i)
                st_async_v2(remote + 8 * i, (uint32_t)o[2 * i], (uint32_t)o[2 * i + 1], rbar);
            mbar_arrive(smem_addr(&ctl->sfull[slot]));
        } else {
            const uint32_t sf = smem_addr(&ctl->sfull[slot]);
            if (!armed) {  // once per use of the slot: this thread's arrival + the description's bytes
                mbar_arrive_expect_tx(sf, (uint32_t)sizeof(TileInfo));
                armed = true;
            }
            if (block) {
                if (!wait_bar(sf, sphase, w, 22, true, true)) return false;
            } else if (!mbar_try_wait_cluster(sf, sphase)) {
                return true;  // not published yet
            }
            ti = ctl->ring[slot];
            mbar_arrive_remote(mapa_shared(smem_addr(&ctl->sempty[slot]), lead));
        }
        armed = false;
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        flag = (ti.e >= 0 && ti.rows > 0 && !p.a_ready && !GATHER) ? ld_acquire_gpu(p.flags + ti.mtile) : w.epoch;
        got = true;
        return true;
    };

    TileInfo cur;
    uint32_t cur_flag = 0;
    bool got = false;
    bool ok = next_tile(cur, cur_flag, true, got);
    bool first = true;
    while (ok && cur.e >= 0) {
        if (p.trace) {
            const unsigned long long t0 = global_timer_ns();
            if (cur.rows > 0 && cur_flag != w.epoch) wait_flag(p.flags + cur.mtile, w, cur.mtile, cur.e);
            const unsigned long long t1 = global_timer_ns();
            trace_add(p, kTrFlagWait, t1 - t0);
            trace_add(p, kTrTiles, 1);
            if (first) trace_set(p, kTrFirstTile, t1);
            first = false;
        } else if (cur.rows > 0 && cur_flag != w.epoch) {
            wait_flag(p.flags + cur.mtile, w, cur.mtile, cur.e);
        }
        fence_proxy_async_global();
        const CUtensorMap* amap = &p.a_map[cur.rank];
        const int brow = cur.e * p.d;
        // this CTA's half of each 256-column MMA: 64-column boxes 4h + {0, 1} (leader) or
        // 4h + {2, 3} (peer) of the tile, for h < kHalves; box b lands at 8192 b in sB
        int bcol[2 * C::kHalves];
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
            for (int b = 0; b < 2; ++b) bcol[2 * h + b] = b_box_col(p, cur.n, C::kBN, 4 * h + (leader ? 0 : 2) + b);
        const int pre_kb = p.k_blocks > kPairClaimKb ? kPairClaimKb : 0;
        TileInfo nxt;
        uint32_t nxt_flag = 0;
        bool have_next = false;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!have_next && kb >= pre_kb) {
                // the leader claims once at pre_kb; the peer polls from pre_kb on
                if (!next_tile(nxt, nxt_flag, false, have_next)) {
                    ok = false;
                    break;
                }
            }
            if (!wait_bar(smem_addr(&ctl->empty[stage]), phase ^ 1u, w, 23, true, true)) {
                ok = false;
                break;
            }
            const uint32_t fb_local = smem_addr(&ctl->full[stage]);
            const uint32_t fb = mapa_shared(fb_local, lead);  // stage barrier of the leader
            if (GATHER) {  // both CTAs' gather warps fill A; the barrier counts the B bytes
                if (leader) mbar_arrive_expect_tx(fb_local, 2 * C::kBBytes);
            } else {
                if (leader) mbar_arrive_expect_tx(fb_local, 2 * C::kStageBytes);
                tma_load_2d_pair(smem_addr(sA + stage * C::kABytes), amap, fb, kb * kTileK, cur.arow);
            }
            if (GATHER) {  // in the dispatch and grouped modes warp 2 issues the B boxes
                if (p.b3d) {  // boxes 2h and 2h + 1 are adjacent chunks: one copy each h
#pragma unroll
                    for (int h = 0; h < C::kHalves; ++h)
                        tma_load_3d_pair(smem_addr(sB + stage * C::kBBytes + 16384 * h), &p.b3_map, fb, 0,
                                         brow + kb * kTileK, bcol[2 * h] >> 6);
                } else {
#pragma unroll
                    for (int b = 0; b < 2 * C::kHalves; ++b)
                        tma_load_2d_pair(smem_addr(sB + stage * C::kBBytes + 8192 * b), &p.b_map, fb,
                                         bcol[b], brow + kb * kTileK);
                }
            }
            last_phase[stage] = (int)phase;
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        if (!have_next && !next_tile(nxt, nxt_flag, true, have_next)) break;
        cur = nxt;
        cur_flag = nxt_flag;
    }
    if (p.trace) trace_set(p, kTrIssueEnd, global_timer_ns());
    // the leader drains its stage barriers: each one completes only when both CTAs'
    // loads of that stage have landed
    if (leader) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s)
            if (last_phase[s] >= 0)
                wait_bar(smem_addr(&ctl->full[s]), (uint32_t)last_phase[s], w, 24, false, true);
    }
}

// B loads of the dispatch and grouped modes (lane 0 of warp 2 of both CTAs of a pair):
// follows the schedule ring like the epilogue and issues this CTA's B boxes of every
// k-block once the stage is free, so the TMA thread issues only A.  A thread issuing a
// k-block's copies is slowed by each one it issues (about 0.26 us per k-block measured for
// three copies), and in this latency-bound pipeline two issuing threads keep the stages
// fuller (Mixtral-shaped dispatch 7% faster).  The leader's TMA thread arms each stage
// for all its bytes; B's may land first (the transaction count goes below zero for a time).
template <int STAGES, int BN>
__device__ void pair_tma_b_role(const DispatchGemmParams& p, SmemCtl* ctl, uint8_t* sB, const Waiter& w,
                                bool leader, uint32_t lead) {
    using C = PairCfg<STAGES, BN>;
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;
    uint32_t sphase = 0;
    for (;;) {
        if (!wait_bar(smem_addr(&ctl->sfull[slot]), sphase, w, 33, true, true)) return;
        const TileInfo ti = ctl->ring[slot];
        const uint32_t se = smem_addr(&ctl->sempty[slot]);
        if (leader) mbar_arrive(se);
        else mbar_arrive_remote(mapa_shared(se, lead));
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        if (ti.e < 0) return;
        int bcol[2 * C::kHalves];
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
            for (int b = 0; b < 2; ++b) bcol[2 * h + b] = b_box_col(p, ti.n, C::kBN, 4 * h + (leader ? 0 : 2) + b);
        const int brow = ti.e * p.d;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!wait_bar(smem_addr(&ctl->empty[stage]), phase ^ 1u, w, 34, true, true)) return;
            const uint32_t fb = mapa_shared(smem_addr(&ctl->full[stage]), lead);
            if (p.b3d) {
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h)
                    tma_load_3d_pair(smem_addr(sB + stage * C::kBBytes + 16384 * h), &p.b3_map, fb, 0,
                                     brow + kb * kTileK, bcol[2 * h] >> 6);
            } else {
#pragma unroll
                for (int b = 0; b < 2 * C::kHalves; ++b)
                    tma_load_2d_pair(smem_addr(sB + stage * C::kBBytes + 8192 * b), &p.b_map, fb, bcol[b],
                                     brow + kb * kTileK);
            }
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

template <int STAGES, int BN, bool GATHER>
__device__ void pair_mma_role(const DispatchGemmParams& p, SmemCtl* ctl, uint8_t* sA, uint8_t* sB,
                              uint32_t tmem_base, const Waiter& w) {
    using C = PairCfg<STAGES, BN>;
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;
    uint32_t sphase = 0;
    int acc = 0;
    uint32_t aphase = 0;
    bool ok = true;
    while (ok) {
        if (!wait_bar(smem_addr(&ctl->sfull[slot]), sphase, w, 25, true, true)) break;
        const int e = ctl->ring[slot].e;
        const uint32_t idesc = ctl->ring[slot].m128 ? C::kIdesc128 : C::kIdesc;
        mbar_arrive(smem_addr(&ctl->sempty[slot]));
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        if (e < 0) break;
        if (!wait_bar(smem_addr(&ctl->tempty[acc]), aphase ^ 1u, w, 26, true, true)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kBN);
        // k-blocks of four K=16 steps in the loop; a last k-block of a reduction that is
        // not a multiple of 64 (fewer steps: the loaded columns past d are not used) after
        // it, so the loop body stays lean (the MMA thread's issue latency is on the
        // critical path)
        const int kfull = p.last_ksteps == kTileK / kUmmaK ? p.k_blocks : p.k_blocks - 1;
        for (int kb = 0; kb < kfull; ++kb) {
            if (!wait_bar(smem_addr(&ctl->full[stage]), phase, w, 27, true, true)) {
                ok = false;
                break;
            }
            if (GATHER) fence_proxy_async_smem();  // this CTA's gathered rows
            tc_fence_after();
            const uint32_t a0 = smem_addr(sA + stage * C::kABytes);
            const uint32_t b0 = smem_addr(sB + stage * C::kBBytes);
#pragma unroll
            for (int kk = 0; kk < kTileK / kUmmaK; ++kk) {
                const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h) {  // tile columns [256h, 256h + 256)
                    const uint64_t bd = smem_desc_sw128(b0 + 16384 * h + kk * 2048, 8192, 1024);
                    umma_bf16_pair(d_tmem + 256u * h, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                }
            }
            umma_commit_pair_mc(smem_addr(&ctl->empty[stage]), 0x3);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (ok && kfull < p.k_blocks) {  // the short last k-block
            if (!wait_bar(smem_addr(&ctl->full[stage]), phase, w, 27, true, true)) break;
            if (GATHER) fence_proxy_async_smem();
            tc_fence_after();
            const uint32_t a0 = smem_addr(sA + stage * C::kABytes);
            const uint32_t b0 = smem_addr(sB + stage * C::kBBytes);
            for (int kk = 0; kk < p.last_ksteps; ++kk) {
                const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h) {
                    const uint64_t bd = smem_desc_sw128(b0 + 16384 * h + kk * 2048, 8192, 1024);
                    umma_bf16_pair(d_tmem + 256u * h, ad, bd, idesc, (kfull | kk) != 0 ? 1u : 0u);
                }
            }
            umma_commit_pair_mc(smem_addr(&ctl->empty[stage]), 0x3);
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        umma_commit_pair_mc(smem_addr(&ctl->tfull[acc]), 0x3);
        if (++acc == C::kAccs) {
            acc = 0;
            aphase ^= 1u;
        }
    }
    umma_commit_pair(smem_addr(&ctl->mma_done));
    wait_bar(smem_addr(&ctl->mma_done), 0u, w, 28, false, true);
}

template <int STAGES, int BN>
__device__ void pair_epilogue_role(const DispatchGemmParams& p, SmemCtl* ctl, uint32_t tmem_base,
                                   const Waiter& w, bool leader, uint32_t lead, float* epi, const int* mt_base) {
    using C = PairCfg<STAGES, BN>;
    const int lane = threadIdx.x & 31;
    const int q = (threadIdx.x >> 5) & 3;
    int slot = 0;
    uint32_t sphase = 0;
    int acc = 0;
    uint32_t aphase = 0;
    for (;;) {
        const bool got = wait_bar(smem_addr(&ctl->sfull[slot]), sphase, w, 29, true, true);
        if (!__all_sync(kFull, got)) break;
        const TileInfo ti = ctl->ring[slot];
        __syncwarp();
        if (lane == 0) {
            const uint32_t se = smem_addr(&ctl->sempty[slot]);
            if (leader) mbar_arrive(se);
            else mbar_arrive_remote(mapa_shared(se, lead));
        }
        if (++slot == kRing) {
            slot = 0;
            sphase ^= 1u;
        }
        if (ti.e < 0) break;
        const bool ready = wait_bar(smem_addr(&ctl->tfull[acc]), aphase, w, 30, true, true);
        if (!__all_sync(kFull, ready)) break;
        tc_fence_after();
        CombineRow cr{0, 0.f, 1};
        if (p.combine) {  // this warp's rows: 32 q + lane, or 32 (q & 1) + lane of an M=128 half
            const int r = ti.m128 ? 32 * (q & 1) + lane : 32 * q + lane;
            cr = combine_row(p, ti.row0, r, ti.rows);
            combine_wait_lower(p, mt_base, true, ti.row0, r, ti.rows, ti.n, cr, w);
            __syncwarp();
        }
        if (ti.m128) {
            epilogue_tile_m128(p, ti, C::kBN, tmem_base + (uint32_t)(acc * C::kBN), q, lane, epi, cr);
        } else if (ti.rows - 32 * q > 0) {  // the odd half of a pair tile may hold fewer rows
            const uint32_t tbase = tmem_base + (uint32_t)(acc * C::kBN) + ((uint32_t)(32 * q) << 16);
            epilogue_tile(p, ti, C::kBN, tbase, q, lane, epi, cr);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            const uint32_t te = smem_addr(&ctl->tempty[acc]);
            if (leader) mbar_arrive(te);
            else mbar_arrive_remote(mapa_shared(te, lead));
        }
        if (p.combine)  // an M=128 tile's two CTAs each publish their 64-row half
            combine_publish(p, ti.rows > 0 ? ti.mtile : -1, ti.n, ti.m128 ? (leader ? 0 : 1) : 0, w.epoch);
        if (++acc == C::kAccs) {
            acc = 0;
            aphase ^= 1u;
        }
    }
}

template <int STAGES, int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    dispatch_gemm_pair_kernel(const __grid_constant__ DispatchGemmParams p) {
    using C = PairCfg<STAGES, BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * C::kABytes;
    float* epi_tiles = reinterpret_cast<float*>(sB + STAGES * C::kBBytes);  // 4 x 32 x 36 fp32
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(reinterpret_cast<uint8_t*>(epi_tiles) + kEpiBytes);
    int* mt_base = reinterpret_cast<int*>(ctl + 1);  // 128-row tiles per expert, prefix
    int* unit_base = mt_base + (kMaxE + 1);           // scatter units per expert, prefix
    int* pt_base = unit_base + (kMaxE + 1);           // 256-row pair tiles per expert, prefix

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank & 1u) == 0u;
    const uint32_t peer = rank ^ 1u;
    const uint32_t lead = rank & ~1u;
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // leader: its expect_tx arrival + both CTAs' bytes (+ its gather warps and the
            // peer's relay in the gather mode); peer's afull: its gather warps
            // gather mode: + the leader's gather threads (on landing) + the peer's relay
            mbar_init(smem_addr(&ctl->full[s]), p.gather ? 1 + 32 * kGatherWarps + 1 : 1);
            mbar_init(smem_addr(&ctl->afull[s]), 32 * kGatherWarps);  // the peer's gather threads
            mbar_init(smem_addr(&ctl->empty[s]), 1);  // the leader's multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_addr(&ctl->tfull[a]), 1);   // the leader's multicast commit
            mbar_init(smem_addr(&ctl->tempty[a]), 8);  // leader: 4 + 4 epilogue warps
        }
        for (int r = 0; r < kRing; ++r) {
            mbar_init(smem_addr(&ctl->sfull[r]), 1);
            // leader: own MMA thread + 4 epilogue warps + the peer's TMA thread and 4 epilogue
            // warps (+ both CTAs' gather warps and the peer's relay in the gather mode)
            mbar_init(smem_addr(&ctl->sempty[r]), 10 + (p.gather ? 2 * kGatherWarps + 1 : 2));
        }
        mbar_init(smem_addr(&ctl->mma_done), 1);
        ctl->abort = 0;
        uint32_t ep = __ldcg(p.hdr + kHdrEpoch) + 1u;
        ctl->epoch = ep == 0u ? 1u : ep;
        mbar_fence_init();
    }
    if (warp == 2) {
        tmem_alloc_pair(smem_addr(&ctl->tmem_base), C::kTmemCols);
        tmem_relinquish_pair();
    }
    build_expert_table(p.offsets, p.E, kTileM, mt_base, ctl->wsum);  // contain __syncthreads
    build_expert_table(p.offsets, p.E, kRowsPerChunk, unit_base, ctl->wsum, p.nch);
    build_expert_table(p.offsets, p.E, 2 * kTileM, pt_base, ctl->wsum);
    if (mt_base[p.E] > p.max_mtiles || __ldg(p.offsets + p.E) != p.T * p.k) {
        __syncthreads();
        if (tid == 0) {
            report_error(p.status, kStDevice, -2, __ldg(p.offsets + p.E), 0);
            for (int e = 0; e <= p.E; ++e) mt_base[e] = pt_base[e] = 0;
            for (int i = 0; i <= p.nch * p.E; ++i) unit_base[i] = 0;
        }
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs running, barrier inits and TMEM address visible to the pair
    tc_fence_after();
    // the pair's role ticket: taken by the leader, written into both CTAs
    if (tid == 0 && leader) {
        const int t = (int)atomicAdd(p.hdr + kHdrRoleCtr, 1u);
        ctl->role = t;
        st_cluster_u32(mapa_shared(smem_addr(&ctl->role), peer), (uint32_t)t);
    }
    cluster_sync_all();
    const uint32_t tmem_base = ctl->tmem_base;
    const uint32_t epoch = ctl->epoch;
    const int scatter_index = 2 * ctl->role + (int)(rank & 1u);
    if (tid == 0 && p.trace) {  // the same thread runs the TMA role: no other writer yet
        for (int i = 0; i < kTraceWords; ++i) trace_set(p, i, 0ull);
        trace_set(p, kTrStart, global_timer_ns());
        trace_set(p, kTrRole, (unsigned long long)ctl->role);
    }

    const long long pipe_timeout = p.timeout_ns * 2 > 500000000LL ? p.timeout_ns * 2 : 500000000LL;
    const Waiter w{&ctl->abort, p.status, p.timeout_ns, pipe_timeout, epoch};
    // the all-warps scatter covers the units before head_units; warp 3 copies the rest
    const int total_units = unit_base[p.nch * p.E];
    int head_units = total_units;
    if (p.bg_head > 0 && p.nch == 1) {
        int h = 0;
        while (h < p.E && pt_base[h] * p.n_tiles < p.bg_head) ++h;
        head_units = unit_base[h];
    }
    if (scatter_index < p.producer_ctas) {
        unsigned long long* w64 = reinterpret_cast<unsigned long long*>(p.hdr);
        if (tid == 0) atomicMax(w64 + kHdrScatterInvStart / 2, ~(unsigned long long)global_timer_ns());
        scatter_role(p, mt_base, unit_base, scatter_index, epoch, sA, ctl, C::kScatterSlots, head_units);
        __syncthreads();
        if (tid == 0) {
            const unsigned long long t = global_timer_ns();
            atomicMax(w64 + kHdrScatterEnd / 2, t);
            trace_set(p, kTrScatterEnd, t);
        }
    }

    if (warp == 0) {
        if (lane == 0) {
            if (p.gather) pair_tma_role<STAGES, BN, true>(p, ctl, mt_base, pt_base, sA, sB, w, leader, peer);
            else pair_tma_role<STAGES, BN, false>(p, ctl, mt_base, pt_base, sA, sB, w, leader, peer);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            if (p.gather) pair_mma_role<STAGES, BN, true>(p, ctl, sA, sB, tmem_base, w);
            else pair_mma_role<STAGES, BN, false>(p, ctl, sA, sB, tmem_base, w);
        }
        else if (lane == 0 && p.gather) pair_relay_role<STAGES>(p, ctl, w, lead);
        __syncwarp();
    } else if (p.gather && warp >= kGatherWarp0 && warp < kGatherWarp0 + kGatherWarps) {
        gather_a_role<STAGES>(p, ctl, sA, w, warp - kGatherWarp0, true, leader, lead);
    } else if (!p.gather && warp == 2) {
        if (lane == 0) pair_tma_b_role<STAGES, BN>(p, ctl, sB, w, leader, lead);
        __syncwarp();
    } else if (warp == 3) {
        if (head_units < total_units) {
            scatter_background(p, mt_base, unit_base, head_units + scatter_index, gridDim.x, total_units, epoch);
            if (lane == 0)
                atomicMax(reinterpret_cast<unsigned long long*>(p.hdr) + kHdrScatterEnd / 2, global_timer_ns());
        }
    } else if (warp >= kEpiWarp0) {
        pair_epilogue_role<STAGES, BN>(p, ctl, tmem_base, w, leader, lead,
                                   epi_tiles + (warp - kEpiWarp0) * kEpiWarpFloats, mt_base);
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 0 && p.trace) trace_set(p, kTrEnd, global_timer_ns());
    cluster_sync_all();  // no CTA leaves while its peer may still signal it
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(p.hdr + kHdrDoneCtr, 1u);
        if (prev == gridDim.x - 1) {
            __threadfence();
            p.hdr[kHdrTileCtr] = 0u;
            p.hdr[kHdrRoleCtr] = 0u;
            p.hdr[kHdrDoneCtr] = 0u;
            p.hdr[kHdrEpoch] = epoch;
            unsigned long long* w64 = reinterpret_cast<unsigned long long*>(p.hdr);
            const unsigned long long inv = atomicExch(w64 + kHdrScatterInvStart / 2, 0ull);
            const unsigned long long end = atomicExch(w64 + kHdrScatterEnd / 2, 0ull);
            w64[kHdrLastScatterStart / 2] = ~inv;
            w64[kHdrLastScatterEnd / 2] = end;
            __threadfence();
        }
    }
}

template <int BN, int STAGES>
cudaError_t launch_cfg(const DispatchGemmParams& p, int grid, size_t smem, cudaStream_t stream) {
    dispatch_gemm_kernel<BN, STAGES><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t dispatch_gemm_pair_smem_bytes(int tile_n) {
    return tile_n == 512 ? PairCfg<4, 512>::kSmem : tile_n == 256 ? PairCfg<6, 256>::kSmem : 0;
}

template <int STAGES, int BN>
cudaError_t pair_prepare(size_t smem, int* max_clusters) {
    cudaError_t e = cudaFuncSetAttribute(dispatch_gemm_pair_kernel<STAGES, BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    return cudaOccupancyMaxActiveClusters(max_clusters, dispatch_gemm_pair_kernel<STAGES, BN>, &cfg);
}

cudaError_t dispatch_gemm_pair_prepare(int tile_n, size_t smem, int* max_clusters) {
    if (tile_n == 512) return pair_prepare<4, 512>(smem, max_clusters);
    if (tile_n == 256) return pair_prepare<6, 256>(smem, max_clusters);
    return cudaErrorInvalidValue;
}

cudaError_t launch_dispatch_gemm_pair(const DispatchGemmParams& p, int grid, size_t smem,
                                      cudaStream_t stream) {
    if (p.tile_n == 512) dispatch_gemm_pair_kernel<4, 512><<<grid, kThreads, smem, stream>>>(p);
    else if (p.tile_n == 256) dispatch_gemm_pair_kernel<6, 256><<<grid, kThreads, smem, stream>>>(p);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

size_t dispatch_gemm_smem_bytes(int tile_n, int stages) {
    if (tile_n == 256 && stages == 4) return Cfg<256, 4>::kSmem;
    if (tile_n == 192 && stages == 4) return Cfg<192, 4>::kSmem;
    if (tile_n == 128 && stages == 6) return Cfg<128, 6>::kSmem;
    return 0;
}

cudaError_t dispatch_gemm_prepare_attributes(int tile_n, int stages, size_t smem) {
    if (tile_n == 256 && stages == 4)
        return cudaFuncSetAttribute(dispatch_gemm_kernel<256, 4>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (tile_n == 192 && stages == 4)
        return cudaFuncSetAttribute(dispatch_gemm_kernel<192, 4>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (tile_n == 128 && stages == 6)
        return cudaFuncSetAttribute(dispatch_gemm_kernel<128, 6>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return cudaErrorInvalidValue;
}

cudaError_t launch_dispatch_gemm(const DispatchGemmParams& p, int grid, int stages, size_t smem,
                                 cudaStream_t stream) {
    if (p.tile_n == 256 && stages == 4) return launch_cfg<256, 4>(p, grid, smem, stream);
    if (p.tile_n == 192 && stages == 4) return launch_cfg<192, 4>(p, grid, smem, stream);
    if (p.tile_n == 128 && stages == 6) return launch_cfg<128, 6>(p, grid, smem, stream);
    return cudaErrorInvalidValue;
}

}  // namespace moe
