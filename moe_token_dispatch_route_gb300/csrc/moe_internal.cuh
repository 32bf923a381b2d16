// Internal declarations shared by the library's translation units: the
// workspace layout, the launch parameter blocks and the sm_103a inline-PTX
// helpers (mbarrier, TMA, tcgen05/TMEM, proxy fences).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- constants

constexpr int kRouteChunk = 64;     // most tokens per routing CTA (8..64, a power of two)
constexpr int kRouteFuseSlots = 8192;  // T*k up to this: the last routing CTA also permutes
// threads of a routing CTA: 8 warps for E <= 32, 16 for more experts (measured: 16 warps
// route the E = 64 and 256 batches 14-18% faster and the E = 8 ones 7-12% slower)
constexpr int route_threads(int E) { return E <= 32 ? 256 : 512; }

constexpr int kTileM = 128;         // GEMM rows per tile (one UMMA M=128)
constexpr int kTileK = 64;          // bf16 elements per 128-byte swizzle row
constexpr int kUmmaK = 16;          // K of one tcgen05.mma kind::f16
constexpr int kRowsPerChunk = 4;    // destination rows per scatter work unit
constexpr int kChunksPerTile = kTileM / kRowsPerChunk;
constexpr int kThreads = 256;       // fused kernel: 8 warps
constexpr int kRing = 8;            // tile-schedule ring entries
constexpr int kMaxRanks = 32;
constexpr int kMaxE = 1024;

// device status codes (same numbers as moe_status_t)
constexpr int kStTimeout = 5;
constexpr int kStCapacity = 6;
constexpr int kStDevice = 7;

// workspace header words (u32)
constexpr int kHdrEpoch = 0;
constexpr int kHdrTileCtr = 8;      // separate 32-byte sectors
constexpr int kHdrRoleCtr = 16;
constexpr int kHdrDoneCtr = 24;
constexpr int kHdrRouteTicket = 32;
constexpr int kHdrScatterInvStart = 40;  // u64: max of ~globaltimer at scatter start (this call)
constexpr int kHdrScatterEnd = 42;       // u64: max of globaltimer at scatter end (this call)
constexpr int kHdrLastScatterStart = 48; // u64: scatter window of the last finished call, ns
constexpr int kHdrLastScatterEnd = 50;   // u64
constexpr size_t kHdrBytes = 256;

struct WorkspaceLayout {
    size_t route_blk_off;   // int32 [route_blocks][E]
    size_t flags_off;       // u32 [max_mtiles]
    size_t chunk_cnt_off;   // u32 [max_mtiles]
    size_t cflags_off;      // u32 [max_mtiles][ceil(N / 128)][2] combine completion words (epoch-tagged)
    size_t total;
};

// ---------------------------------------------------------------- launches

struct RouteArgs {
    const float* logits;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* dest;
    uint32_t* hdr;
    int32_t* blk;     // [nb][E] per-CTA counts, then per-CTA bases
    int T, E, k, nb;
    int chunk;        // tokens per CTA (set by launch_route)
    int fuse_permute; // 1: the last CTA also writes dest and perm (set by launch_route)
    const float* sel_bias;  // [E] added to the logits for selection only; nullptr: none
    int renorm;       // 1: each token's gates are divided by their sum over the k picks
    int sigmoid;      // 1: gate score = logistic(logit); 0: softmax over all E
};

// Routing CTAs for T tokens and E experts: tokens per CTA is the smallest of 8, 16,
// 32, 64 that keeps the CTA count within max(SM count, kRouteScanEntries / E) (64
// when none does).
constexpr int kRouteScanEntries = 4096;
int route_blocks_for(int T, int E, int sm_count);
cudaError_t launch_route(const RouteArgs& a, cudaStream_t stream);
cudaError_t route_prepare_attributes();

struct DispatchGemmParams {
    CUtensorMap a_map[kMaxRanks];   // rank receive buffers, bf16 [cap][d], box 64 x 128
    CUtensorMap b_map;              // W viewed as bf16 [E*d][N], box 64 x 64
    CUtensorMap b3_map;             // W as 64-column chunks: dims {64, E*d, N/64}, box 64 x 64 x 2
    int b3d;                        // 1: B boxes are loaded two chunks at a time through b3_map
    const uint16_t* x;
    const int32_t* offsets;
    const int32_t* perm;
    uint16_t* recv[kMaxRanks];
    void* Y;                        // fp32, or bf16 when out_bf16
    uint32_t* hdr;
    uint32_t* flags;
    uint32_t* chunk_cnt;
    int32_t* status;
    long long timeout_ns;
    int T, d, E, k, N, R, cap;
    int tile_n, n_tiles, k_blocks;  // k_blocks = ceil(d / 64)
    int last_ksteps;                // K=16 MMA steps in the last k-block: (d - 64 (k_blocks - 1)) / 16
    int producer_ctas;
    int max_mtiles;                 // size of flags[] and chunk_cnt[]
    int skip_publish;               // m-tile whose flag is never published, or -1
    int band;                       // row tiles per schedule band; 0 = the whole expert
    int half_tiles;                 // single CTAs: 0 whole tiles only; 1 every tile as two half-width
                                    //   tiles when the schedule has at most gridDim/2 tiles; 2 always
    int nch;                        // scatter order: parts per expert, chunk-major (nch E <= 1024)
    int bg_head;                    // CTA pairs: > 0: every warp scatters only the rows of the first
                                    //   experts holding at least bg_head pair tiles before the GEMM,
                                    //   warp 3 the rest beside it (expert-major, nch 1); 0: all first
    int glu;                        // 1: W = [gate | up], each F = N/2 wide; out H, not Y
    int F;                          // N/2 when glu
    uint16_t* H;                    // glu: bf16 [S][F], silu(gate) * up
    int a_ready;                    // 1: A rows are already in a_map[0] (no scatter, no flags)
    int gather;                     // 1: A rows are copied from x by perm into shared memory
                                    //    (no receive buffers, no scatter, no flags)
    int out_bf16;                   // 1: Y is bf16 (fp32 accumulator rounded once)
    int combine;                    // 1: no Y; each row, times its slot's gate, goes into its
                                    //    token's row of `out`: stored by the token's lowest
                                    //    expert, then added by the others in expert order
    const float* topk_w;            // combine: [T*k] gate of each slot
    const int32_t* dest;            // combine: [T*k] destination row of each slot
    float* out;                     // combine: fp32 [T][N]
    uint32_t* cflags;               // combine: u32 [max_mtiles][n_tiles][2] tile completion words
    unsigned long long* trace;      // [grid][kTraceWords] per-CTA stamps, or null (off)
};

// Per-CTA trace record (moe_set_trace): global-timer stamps in ns and counters.
constexpr int kTraceWords = 8;
constexpr int kTrStart = 0;      // CTA past its setup
constexpr int kTrScatterEnd = 1; // CTA finished its scatter share (0: no scatter role)
constexpr int kTrFirstTile = 2;  // TMA thread: first tile's rows ready (after its flag)
constexpr int kTrFlagWait = 3;   // TMA thread: total ns waiting for ready flags
constexpr int kTrTiles = 4;      // TMA thread: tiles this CTA loaded (pair tiles count once per CTA)
constexpr int kTrIssueEnd = 5;   // TMA thread: last load issued
constexpr int kTrEnd = 6;        // CTA done with its roles
constexpr int kTrRole = 7;       // role ticket

cudaError_t launch_dispatch_gemm(const DispatchGemmParams& p, int grid, int stages,
                                 size_t smem, cudaStream_t stream);
size_t dispatch_gemm_smem_bytes(int tile_n, int stages);
struct RouterArgs {
    const uint16_t* x;   // bf16 [T][d]
    const uint16_t* Wr;  // bf16 [d][E]
    const float* bias;   // fp32 [E] or null
    float* L;            // fp32 [T][E]
    int T, d, E;
    int sm_count;
};
cudaError_t launch_router_logits(const RouterArgs& a, cudaStream_t stream);
cudaError_t router_prepare_attributes();  // shared-memory opt-in of the router kernels

struct CombineArgs {
    const void* Y;        // [S][N] destination order, fp32 or bf16
    int y_bf16;
    const float* w;       // [T][k] gate weights
    const int32_t* dest;  // [T*k]
    float* out;           // [T][N]
    int T, k, N, S;
};
cudaError_t launch_combine(const CombineArgs& a, int sm_count, cudaStream_t stream);

// CTA-pair mode (clusters of 2, 256 x 256 tiles, tcgen05 cta_group::2)
size_t dispatch_gemm_pair_smem_bytes(int tile_n);  // tile_n: 256 or 512
cudaError_t dispatch_gemm_pair_prepare(int tile_n, size_t smem, int* max_clusters);
cudaError_t launch_dispatch_gemm_pair(const DispatchGemmParams& p, int grid, size_t smem,
                                      cudaStream_t stream);
cudaError_t dispatch_gemm_prepare_attributes(int tile_n, int stages, size_t smem);

// ---------------------------------------------------------------- PTX helpers

#if defined(__CUDACC__)

// 16-byte read-only load that does not allocate in L1
__device__ __forceinline__ uint4 ld_nc_na_v4(const uint4* ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// first error wins; later ones are dropped
__device__ __forceinline__ void report_error(int32_t* status, int code, int a0, int a1, int a2) {
    if (atomicCAS(status, 0, code) == 0) {
        status[1] = a0;
        status[2] = a1;
        status[3] = a2;
    }
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// orders this thread's generic-proxy global accesses with its async-proxy (TMA) ones
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- cp.async (16-byte global -> shared, bypassing L1; per-thread commit groups)

__device__ __forceinline__ void cp_async16_cg(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// src_bytes (0 or 16) bytes are read; the rest of the 16 are filled with zeros
__device__ __forceinline__ void cp_async16_cg_zfill(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// one arrival on a barrier of this CTA once every cp.async this thread has issued so
// far has landed (.noinc: the barrier's expected count includes this arrival)
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// waits until at most n (0..7) of this thread's cp.async groups are pending
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
    switch (n) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        default: cp_async_wait<7>(); break;
    }
}

// ---- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---- TMA (tensor, tiled, global -> shared, completes on an mbarrier)

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// ---- tcgen05 / TMEM

__device__ __forceinline__ void tmem_alloc(uint32_t holder_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(holder_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]; bf16 inputs, fp32 accumulator, one thread issues
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// the mbarrier gets one arrival once every earlier tcgen05 op of this thread is done
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}

// 32 TMEM lanes x 32 consecutive 32-bit columns; thread i of the warp gets lane (base + i)
__device__ __forceinline__ void tmem_ld_32x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// waits for this thread's tcgen05.ld; the registers are tied in so no use moves above it
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Shared-memory matrix descriptor of tcgen05.mma, 128-byte swizzle:
// bits 0-13 start address >> 4, 16-29 leading byte offset >> 4,
// 32-45 stride byte offset >> 4, 46-48 = 0b001, 49-51 base offset (0: the
// swizzle atoms are 1024-byte aligned), 61-63 layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// ---- CTA pairs (clusters of 2) for tcgen05 cta_group::2

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t smem, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem), "r"(rank));
    return r;
}

// all threads of both CTAs; orders earlier shared-memory writes (local or remote) before later reads
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// arrive on an mbarrier given by its shared::cluster address (this CTA or the peer)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// arrive on the peer CTA's mbarrier with release semantics at CTA scope: the form for a
// signal that hands a buffer (a stage, a ring slot, an accumulator) back or on, where the
// data itself needs no cluster-scope ordering (the cluster-scope release above costs about
// a microsecond per arrival, measured)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// 8 bytes into the peer CTA's shared memory, counted as 8 transaction bytes on the peer's
// mbarrier `mbar_cluster` once they are visible there
__device__ __forceinline__ void st_async_v2(uint32_t addr_cluster, uint32_t a, uint32_t b, uint32_t mbar_cluster) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];"
                 ::"r"(addr_cluster), "r"(a), "r"(b), "r"(mbar_cluster) : "memory");
}

// wait on a local mbarrier whose arrivals may come from the peer CTA
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// TMA tile load whose completion is signalled on an mbarrier of either CTA of the pair
// Two adjacent 64-column chunks of W in one copy (3-D map {64, rows, chunks}, box
// 64 x 64 x 2): they land as two 8 KB 128-byte-swizzled boxes, one after the other.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

// one warp in each CTA of the pair allocates the same columns in both TMEMs
__device__ __forceinline__ void tmem_alloc_pair(uint32_t holder_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(holder_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// issued by one thread of the even CTA: D (256 rows, half in each CTA's TMEM) (+)= A (128 rows
// from each CTA's shared memory) * B (N/2 columns from each CTA's shared memory)
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// one arrival, once the issuing thread's earlier tcgen05 ops are done, on the mbarrier at
// the same shared-memory offset in every CTA of `mask`
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(bar), "h"(mask) : "memory");
}

__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}

#endif  // __CUDACC__

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, 10-12 = 1), A K-major (bit 15 = 0), B MN-major
// (bit 16 = 1), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t idesc_bf16_f32_kmajA_mnmajB(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace moe
