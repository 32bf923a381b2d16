// C ABI of the library (declared in include/moe.h): argument validation,
// the plan (tile configuration and role split), TMA tensor-map encoding and
// the launches.  Host code only; the kernels live in route.cu and
// dispatch_gemm.cu.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "moe.h"
#include "moe_internal.cuh"

using namespace moe;

struct moe_plan_s {
    moe_shape_t shape;
    int device = 0;
    int sm_count = 0;
    int T = 0, d = 0, E = 0, k = 0, N = 0, R = 1, cap = 0;
    long long S = 0;
    int tile_n = 256, stages = 4, num_ctas = 0, producer_ctas = 0;
    int max_mtiles = 0, route_blocks = 0;
    size_t smem = 0;
    WorkspaceLayout ws{};
    long long timeout_ns = 0;
    int skip_publish = -1;
    int band = 0;
    int half_tiles = 0;  // single-CTA plans: 1 = small schedules run as half-width tiles
    int bg_head = -1;    // CTA pairs: pair tiles the all-warps scatter covers before the GEMM
                         //   (the rest is copied beside it); -1 auto by output width, 0 off
    int scatter_parts = 1;  // scatter order: parts per expert (chunk-major), nch E <= kMaxE
    bool pair = false;  // CTA-pair mode: clusters of 2, 256 x 256 tiles, tcgen05 cta_group::2
    unsigned long long* trace = nullptr;  // per-CTA trace records (moe_set_trace), or null
    // tensor maps, re-encoded only when the buffers change
    std::mutex mu;
    bool maps_valid = false;
    const void* map_W = nullptr;
    int map_nA = 0;          // A buffers encoded: R receive buffers, or 1 caller buffer
    uint64_t map_rows = 0;   // rows of each A buffer
    const void* map_A[kMaxRanks] = {};
    CUtensorMap a_maps[kMaxRanks];
    CUtensorMap b_map;
    CUtensorMap b3_map;  // W as 64-column chunks (valid when b3_ok)
    bool b3_ok;
};

namespace {

constexpr long long kDefaultTimeoutNs = 2000000000LL;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Makes `dev` current for the duration of a call and restores the previous device.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            prev = -1;
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// bf16 [rows][cols] row-major, 128-byte swizzle, box = box_cols x box_rows
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_cols, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// W [rows][cols] bf16 (cols % 64 == 0) as 64-column chunks: dims {64, rows, cols/64}
// with strides {cols*2, 128} bytes, box 64 x 64 x 2, 128-byte swizzle: one copy moves
// two adjacent chunks, landing exactly as two boxes of the 2-D map one after the other.
bool encode_bf16_chunks(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
    auto enc = tensor_map_encoder();
    if (!enc || cols % 64 != 0) return false;
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64, 64, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

moe_status_t validate_shape(const moe_shape_t& s) {
    if (s.T < 0 || s.d <= 0 || s.E <= 0 || s.k <= 0 || s.N <= 0 || s.num_ranks < 0 ||
        s.rank_capacity_rows < 0 || s.producer_ctas < 0 || s.num_ctas < 0 || s.timeout_ns < 0 ||
        s.debug_skip_publish < 0 || (s.route_flags & ~(MOE_ROUTE_RENORM | MOE_ROUTE_SIGMOID)) != 0 ||
        (s.out_dtype != MOE_OUT_F32 && s.out_dtype != MOE_OUT_BF16))
        return MOE_ERR_INVALID_ARG;
    const int R = s.num_ranks == 0 ? 1 : s.num_ranks;
    if (s.E > kMaxE || s.k > std::min(s.E, 32)) return MOE_ERR_UNSUPPORTED;
    if (s.d % kUmmaK != 0 || s.d > 65536) return MOE_ERR_UNSUPPORTED;  // whole K=16 MMA steps
    if (s.N % 16 != 0) return MOE_ERR_UNSUPPORTED;
    if (R > kMaxRanks || s.E % R != 0) return MOE_ERR_UNSUPPORTED;
    if ((long long)s.T * s.k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    if (s.tile_n != 0 && s.tile_n != 128 && s.tile_n != 192 && s.tile_n != 256 && s.tile_n != 512)
        return MOE_ERR_UNSUPPORTED;
    if (s.tile_m != 0 && s.tile_m != 128 && s.tile_m != 256) return MOE_ERR_UNSUPPORTED;
    if (s.tile_m == 256 && (s.N < 256 || (s.tile_n != 0 && s.tile_n != 256 && s.tile_n != 512)))
        return MOE_ERR_UNSUPPORTED;
    if (s.tile_n == 512 && (s.tile_m == 128 || s.N < 512)) return MOE_ERR_UNSUPPORTED;  // pairs only
    return MOE_OK;
}

}  // namespace

namespace moe {
// Shape fields the routing launch needs, for entry points defined in other files.
bool plan_route_shape(moe_plan_t plan, int* T, int* E, int* k, int* route_blocks, int* device,
                      int* route_flags) {
    if (!plan) return false;
    *route_flags = plan->shape.route_flags;
    *T = plan->T;
    *E = plan->E;
    *k = plan->k;
    *route_blocks = plan->route_blocks;
    *device = plan->device;
    return true;
}
}  // namespace moe

// CTA pairs on wide layers: every warp scatters only the rows of the first experts that hold
// the first two waves of pair tiles (num_ctas pair tiles), then joins the GEMM, while warp 3 of
// every CTA copies the remaining rows beside it.  A GEMM of `out_cols` output columns needs
// out_cols flops per byte of A, so at the bf16 peak a layer of at least kBgMinCols columns
// consumes rows at under 0.25 TB/s, which those warps (about 0.3 TB/s measured) keep ahead
// of; narrower layers scatter everything first.  Returns the head in pair tiles, 0 off.
constexpr int kBgMinCols = 8192;
static int bg_head_for(const moe_plan_s* plan, int out_cols) {
    if (!plan->pair) return 0;
    if (plan->bg_head >= 0) return plan->bg_head;
    return out_cols >= kBgMinCols ? plan->num_ctas : 0;
}

extern "C" {

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
        case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    }
    return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_plan(const moe_shape_t* shape, int device, moe_plan_t* plan, size_t* workspace_bytes) {
    if (!shape || !plan || !workspace_bytes || device < 0) return MOE_ERR_INVALID_ARG;
    *plan = nullptr;
    moe_status_t st = validate_shape(*shape);
    if (st != MOE_OK) return st;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    DeviceGuard guard(device);
    if (!guard.ok) return MOE_ERR_CUDA;
    int major = 0, minor = 0, sms = 0, smem_optin = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only

    moe_plan_s* p = new (std::nothrow) moe_plan_s();
    if (!p) return MOE_ERR_INVALID_ARG;
    p->shape = *shape;
    p->device = device;
    p->sm_count = sms;
    p->T = shape->T;
    p->d = shape->d;
    p->E = shape->E;
    p->k = shape->k;
    p->N = shape->N;
    p->R = shape->num_ranks == 0 ? 1 : shape->num_ranks;
    p->S = (long long)p->T * p->k;
    p->cap = shape->rank_capacity_rows == 0 ? (int)p->S : shape->rank_capacity_rows;
    // single-CTA tile width (512-wide tiles exist for CTA pairs only)
    p->tile_n = shape->tile_n != 0 && shape->tile_n != 512 ? shape->tile_n : (p->N >= 256 ? 256 : 128);
    p->stages = p->tile_n == 128 ? 6 : 4;
    p->smem = dispatch_gemm_smem_bytes(p->tile_n, p->stages);
    if (p->smem == 0 || (int)p->smem > smem_optin) {
        delete p;
        return MOE_ERR_UNSUPPORTED;
    }
    p->num_ctas = shape->num_ctas != 0 ? std::min(shape->num_ctas, sms) : sms;
    // CTA pairs for layers with many rows per expert (on average at least one 256-row
    // tile) and full-width tiles, unless the shape fixes tile_m
    if (shape->tile_m == 0)
        p->pair = p->S >= 256LL * p->E && p->N >= 256 &&
                  (shape->tile_n == 0 || shape->tile_n == 256 || shape->tile_n == 512);
    else
        p->pair = shape->tile_m == 256;
    if (p->pair) {
        const int pair_tn = shape->tile_n == 512 ? 512 : 256;
        int max_clusters = 0;
        p->smem = dispatch_gemm_pair_smem_bytes(pair_tn);
        if ((int)p->smem > smem_optin ||
            dispatch_gemm_pair_prepare(pair_tn, p->smem, &max_clusters) != cudaSuccess || max_clusters < 1) {
            cudaGetLastError();
            if (shape->tile_m == 256 || shape->tile_n == 512) {  // pairs were asked for and cannot run here
                delete p;
                return MOE_ERR_UNSUPPORTED;
            }
            p->pair = false;  // no co-resident pairs: keep the single-CTA kernel
            p->smem = dispatch_gemm_smem_bytes(p->tile_n, p->stages);
        } else {
            p->tile_n = pair_tn;
            p->stages = pair_tn == 512 ? 4 : 6;
            p->num_ctas = 2 * std::min(max_clusters, p->num_ctas / 2);
        }
    } else if (shape->tile_n == 512) {
        delete p;
        return MOE_ERR_UNSUPPORTED;
    }
    // Every CTA starts in the scatter role by default: the scatter then ends soonest and
    // the first tiles' flags come earliest.  Measured against 16-96 scatter CTAs this is
    // the fastest or within 0.5% on the Mixtral-, fine-grained-, DeepSeek-V3-shaped and
    // decode layers (up to 4.5% faster on the decode batch).
    const int auto_p = p->num_ctas;
    p->producer_ctas = shape->producer_ctas != 0 ? shape->producer_ctas : auto_p;
    p->producer_ctas = std::max(1, std::min(p->producer_ctas, p->num_ctas));
    if (p->pair) p->producer_ctas = std::min(p->num_ctas, (p->producer_ctas + 1) & ~1);  // whole pairs
    p->max_mtiles = (int)(p->S / kTileM) + p->E;
    p->route_blocks = route_blocks_for(p->T, p->E, sms);
    p->timeout_ns = shape->timeout_ns != 0 ? shape->timeout_ns : kDefaultTimeoutNs;
    p->skip_publish = shape->debug_skip_publish > 0 ? shape->debug_skip_publish - 1 : -1;
    // tuning override for sweeps only: row tiles per schedule band (0 = whole expert)
    if (const char* env = std::getenv("MOE_TILE_BAND")) p->band = std::max(0, std::atoi(env));
    // A schedule with fewer tiles than half the CTAs (a small, latency-bound layer) leaves
    // most SMs idle; there every single-CTA tile is claimed as two half-width tiles, left
    // and right, which the kernel decides once routing has fixed the tile count.  Halves
    // need whole 64-column boxes: BN 128 or 256.  (Splitting the last wave of a large
    // HBM-bound layer instead was measured slower: a half carries the whole A traffic.)
    if (!p->pair && (p->tile_n == 128 || p->tile_n == 256)) p->half_tiles = 1;
    if (const char* env = std::getenv("MOE_HALF_TILES"))  // tuning override: 0 never, 2 always
        p->half_tiles = p->half_tiles ? std::max(0, std::min(2, std::atoi(env))) : 0;
    // tuning override for sweeps and tests: the background scatter's head (0 off)
    if (const char* env = std::getenv("MOE_BG_HEAD")) p->bg_head = std::max(0, std::atoi(env));
    // The scatter walks each expert's rows in token-ordered parts of about 1024 tokens (at
    // most 16), part-major, so that a token's k copies are made while its x row is in L2.
    p->scatter_parts = std::max(1, std::min(std::min(16, kMaxE / p->E), p->T / 1024));
    if (const char* env = std::getenv("MOE_SCATTER_PARTS"))  // tuning override for sweeps only
        p->scatter_parts = std::max(1, std::min(std::atoi(env), kMaxE / p->E));

    size_t off = kHdrBytes;
    p->ws.route_blk_off = off;
    off = round_up(off + (size_t)std::max(1, p->route_blocks) * p->E * 4, 256);
    p->ws.flags_off = off;
    off = round_up(off + (size_t)p->max_mtiles * 4, 256);
    p->ws.chunk_cnt_off = off;
    off = round_up(off + (size_t)p->max_mtiles * 4, 256);
    p->ws.cflags_off = off;
    off = round_up(off + (size_t)p->max_mtiles * ((p->N + kTileM - 1) / kTileM) * 2 * 4, 256);
    p->ws.total = off;

    if ((!p->pair && dispatch_gemm_prepare_attributes(p->tile_n, p->stages, p->smem) != cudaSuccess) ||
        route_prepare_attributes() != cudaSuccess || router_prepare_attributes() != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return MOE_ERR_CUDA;
    }
    *plan = p;
    *workspace_bytes = p->ws.total;
    return MOE_OK;
}

moe_status_t moe_plan_destroy(moe_plan_t plan) {
    delete plan;
    return MOE_OK;
}

moe_status_t moe_plan_info(moe_plan_t plan, moe_plan_info_t* info) {
    if (!plan || !info) return MOE_ERR_INVALID_ARG;
    info->tile_m = plan->pair ? 2 * kTileM : kTileM;
    info->tile_n = plan->tile_n;
    info->tile_k = kTileK;
    info->stages = plan->stages;
    info->num_ctas = plan->num_ctas;
    info->producer_ctas = plan->producer_ctas;
    info->sm_count = plan->sm_count;
    info->smem_bytes = (int32_t)plan->smem;
    info->max_mtiles = plan->max_mtiles;
    info->route_blocks = plan->route_blocks;
    info->workspace_bytes = (int64_t)plan->ws.total;
    info->half_tiles = plan->half_tiles;
    info->background_scatter = bg_head_for(plan, plan->N);
    return MOE_OK;
}

moe_status_t moe_route(moe_plan_t plan, const float* logits, int32_t* topk_idx, float* topk_w,
                       int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* dest,
                       void* workspace, void* stream) {
    return moe_route_biased(plan, logits, nullptr, topk_idx, topk_w, counts, offsets, perm, dest,
                            workspace, stream);
}

moe_status_t moe_route_biased(moe_plan_t plan, const float* logits, const float* selection_bias,
                              int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                              int32_t* perm, int32_t* dest, void* workspace, void* stream) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    if (selection_bias && !aligned(selection_bias, 4)) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || !aligned(counts, 4) || !aligned(offsets, 4))
        return MOE_ERR_INVALID_ARG;
    if (plan->T > 0 && (!logits || !topk_idx || !topk_w || !perm || !dest ||
                        !aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
                        !aligned(perm, 4) || !aligned(dest, 4)))
        return MOE_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256)) return MOE_ERR_WORKSPACE;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan->T == 0) {
        if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * plan->E, s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (plan->E + 1), s) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        return MOE_OK;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    RouteArgs a;
    a.logits = logits;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    a.dest = dest;
    a.hdr = reinterpret_cast<uint32_t*>(ws);
    a.blk = reinterpret_cast<int32_t*>(ws + plan->ws.route_blk_off);
    a.T = plan->T;
    a.E = plan->E;
    a.k = plan->k;
    a.nb = plan->route_blocks;
    a.sel_bias = selection_bias;
    a.renorm = (plan->shape.route_flags & MOE_ROUTE_RENORM) ? 1 : 0;
    a.sigmoid = (plan->shape.route_flags & MOE_ROUTE_SIGMOID) ? 1 : 0;
    if (launch_route(a, s) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

}  // extern "C"

namespace {

enum class GemmMode { kDispatch, kDispatchSwiglu, kGrouped, kGather, kDispatchCombine };

// The three entry points that run the persistent GEMM kernel.  kDispatch and
// kDispatchSwiglu scatter x into the receive buffers and compute on the rows
// as they land; kGrouped computes on rows the caller has already laid out.
moe_status_t run_gemm(moe_plan_t plan, GemmMode mode, const uint16_t* x, const int32_t* offsets,
                      const int32_t* perm, const uint16_t* W, void* const* recv, const uint16_t* A,
                      void* Y, uint16_t* H, void* workspace, int32_t* dev_status, void* stream,
                      const int32_t* dest = nullptr, const float* topk_w = nullptr, float* out = nullptr) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    if (!dev_status || !aligned(dev_status, 4)) return MOE_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256)) return MOE_ERR_WORKSPACE;
    const bool glu = mode == GemmMode::kDispatchSwiglu;
    const bool combine = mode == GemmMode::kDispatchCombine;
    if (glu && plan->tile_n == 192) return MOE_ERR_UNSUPPORTED;  // halves must be whole 64-column boxes
    if (plan->T == 0) return MOE_OK;
    if (!offsets || !W || !aligned(W, 16) || !aligned(offsets, 4)) return MOE_ERR_INVALID_ARG;
    if (combine) {
        if (!dest || !topk_w || !out || !aligned(dest, 4) || !aligned(topk_w, 4) || !aligned(out, 16))
            return MOE_ERR_INVALID_ARG;
    } else if (glu ? (!H || !aligned(H, 16)) : (!Y || !aligned(Y, 16))) {
        return MOE_ERR_INVALID_ARG;
    }
    const bool grouped = mode == GemmMode::kGrouped;
    const bool gather = mode == GemmMode::kGather;
    const int nA = grouped ? 1 : gather ? 0 : plan->R;  // A tensor maps (the gather has none)
    const void* abuf[kMaxRanks] = {};
    if (grouped) {
        if (!A || !aligned(A, 16)) return MOE_ERR_INVALID_ARG;
        abuf[0] = A;
    } else if (gather) {
        if (!x || !perm || !aligned(x, 16) || !aligned(perm, 4)) return MOE_ERR_INVALID_ARG;
    } else {
        if (!x || !perm || !recv || !aligned(x, 16) || !aligned(perm, 4)) return MOE_ERR_INVALID_ARG;
        for (int r = 0; r < plan->R; ++r) {
            if (!recv[r] || !aligned(recv[r], 16)) return MOE_ERR_INVALID_ARG;
            abuf[r] = recv[r];
        }
    }
    const uint64_t arows = grouped ? (uint64_t)plan->S : (uint64_t)plan->cap;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return MOE_ERR_CUDA;

    DispatchGemmParams prm;
    {
        std::lock_guard<std::mutex> lock(plan->mu);
        bool same = plan->maps_valid && plan->map_W == W && plan->map_nA == nA && plan->map_rows == arows;
        for (int r = 0; same && r < nA; ++r) same = plan->map_A[r] == abuf[r];
        if (!same) {
            plan->maps_valid = false;
            for (int r = 0; r < nA; ++r)
                if (!encode_bf16_2d(&plan->a_maps[r], abuf[r], arows, (uint64_t)plan->d, kTileK, kTileM))
                    return MOE_ERR_CUDA;
            if (!encode_bf16_2d(&plan->b_map, W, (uint64_t)plan->E * plan->d, (uint64_t)plan->N, 64,
                                kTileK))
                return MOE_ERR_CUDA;
            // the chunked view is an optimisation: where it cannot be encoded the 2-D map serves
            plan->b3_ok = encode_bf16_chunks(&plan->b3_map, W, (uint64_t)plan->E * plan->d, (uint64_t)plan->N);
            plan->map_W = W;
            plan->map_nA = nA;
            plan->map_rows = arows;
            for (int r = 0; r < nA; ++r) plan->map_A[r] = abuf[r];
            plan->maps_valid = true;
        }
        std::memset(&prm, 0, sizeof prm);
        for (int r = 0; r < nA; ++r) prm.a_map[r] = plan->a_maps[r];
        prm.b_map = plan->b_map;
        prm.b3_map = plan->b3_map;
        // chunk pairs must start on a chunk boundary: N % 64 == 0, and F % 64 == 0 for the
        // gated layout (its up half starts at column F)
        prm.b3d = (plan->b3_ok && (!glu || (plan->N / 2) % 64 == 0)) ? 1 : 0;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    prm.x = x;
    prm.offsets = offsets;
    prm.perm = perm;
    if (!grouped && !gather)  // the gather mode has no receive buffers (recv may be NULL)
        for (int r = 0; r < plan->R; ++r) prm.recv[r] = static_cast<uint16_t*>(recv[r]);
    prm.Y = Y;
    prm.out_bf16 = (!combine && plan->shape.out_dtype == MOE_OUT_BF16) ? 1 : 0;
    prm.combine = combine ? 1 : 0;
    prm.topk_w = topk_w;
    prm.dest = dest;
    prm.out = out;
    prm.trace = plan->trace;
    prm.H = H;
    prm.glu = glu ? 1 : 0;
    prm.F = plan->N / 2;
    prm.a_ready = grouped ? 1 : 0;
    prm.gather = gather ? 1 : 0;
    prm.hdr = reinterpret_cast<uint32_t*>(ws);
    prm.flags = reinterpret_cast<uint32_t*>(ws + plan->ws.flags_off);
    prm.chunk_cnt = reinterpret_cast<uint32_t*>(ws + plan->ws.chunk_cnt_off);
    prm.cflags = reinterpret_cast<uint32_t*>(ws + plan->ws.cflags_off);
    prm.status = dev_status;
    prm.timeout_ns = plan->timeout_ns;
    prm.T = plan->T;
    prm.d = plan->d;
    prm.E = plan->E;
    prm.k = plan->k;
    prm.N = plan->N;
    prm.R = (grouped || gather) ? 1 : plan->R;
    prm.cap = (grouped || gather) ? (int)plan->S : plan->cap;
    prm.tile_n = plan->tile_n;
    const int tile_cols = glu ? plan->tile_n / 2 : plan->tile_n;  // output columns per tile
    const int out_cols = glu ? plan->N / 2 : plan->N;
    prm.n_tiles = (out_cols + tile_cols - 1) / tile_cols;
    prm.k_blocks = (plan->d + kTileK - 1) / kTileK;
    prm.last_ksteps = (plan->d - kTileK * (prm.k_blocks - 1)) / kUmmaK;
    prm.producer_ctas = (grouped || gather) ? 0 : plan->producer_ctas;
    prm.max_mtiles = plan->max_mtiles;
    prm.skip_publish = plan->skip_publish;
    prm.band = plan->band;
    // gated and combining epilogues keep whole tiles (their column bookkeeping is per tile)
    prm.half_tiles = (glu || combine) ? 0 : plan->half_tiles;
    prm.nch = plan->scatter_parts;
    prm.bg_head = (grouped || gather) ? 0 : bg_head_for(plan, out_cols);
    if (prm.bg_head > 0) prm.nch = 1;  // the head is a prefix of experts: expert-major walk
    cudaError_t lerr;
    if (plan->pair) {
        lerr = launch_dispatch_gemm_pair(prm, plan->num_ctas, plan->smem, static_cast<cudaStream_t>(stream));
    } else {
        lerr = launch_dispatch_gemm(prm, plan->num_ctas, plan->stages, plan->smem,
                                    static_cast<cudaStream_t>(stream));
    }
    if (lerr != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_dispatch_gemm(moe_plan_t plan, const uint16_t* x, const int32_t* offsets,
                               const int32_t* perm, const uint16_t* W, void* const* recv, void* Y,
                               void* workspace, int32_t* dev_status, void* stream) {
    return run_gemm(plan, GemmMode::kDispatch, x, offsets, perm, W, recv, nullptr, Y, nullptr,
                    workspace, dev_status, stream);
}

moe_status_t moe_dispatch_gemm_combine(moe_plan_t plan, const uint16_t* x, const int32_t* offsets,
                                       const int32_t* perm, const int32_t* dest, const float* topk_w,
                                       const uint16_t* W, void* const* recv, float* out, void* workspace,
                                       int32_t* dev_status, void* stream) {
    return run_gemm(plan, GemmMode::kDispatchCombine, x, offsets, perm, W, recv, nullptr, nullptr, nullptr,
                    workspace, dev_status, stream, dest, topk_w, out);
}

moe_status_t moe_dispatch_gemm_swiglu(moe_plan_t plan, const uint16_t* x, const int32_t* offsets,
                                      const int32_t* perm, const uint16_t* W1, void* const* recv,
                                      uint16_t* H, void* workspace, int32_t* dev_status,
                                      void* stream) {
    return run_gemm(plan, GemmMode::kDispatchSwiglu, x, offsets, perm, W1, recv, nullptr, nullptr, H,
                    workspace, dev_status, stream);
}

moe_status_t moe_gather_gemm(moe_plan_t plan, const uint16_t* x, const int32_t* offsets,
                             const int32_t* perm, const uint16_t* W, void* Y, void* workspace,
                             int32_t* dev_status, void* stream) {
    return run_gemm(plan, GemmMode::kGather, x, offsets, perm, W, nullptr, nullptr, Y, nullptr,
                    workspace, dev_status, stream);
}

moe_status_t moe_grouped_gemm(moe_plan_t plan, const uint16_t* A, const int32_t* offsets,
                              const uint16_t* W, void* Y, void* workspace, int32_t* dev_status,
                              void* stream) {
    return run_gemm(plan, GemmMode::kGrouped, nullptr, offsets, nullptr, W, nullptr, A, Y, nullptr,
                    workspace, dev_status, stream);
}

moe_status_t moe_set_trace(moe_plan_t plan, void* trace, int64_t bytes) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    if (!trace) {
        plan->trace = nullptr;
        return MOE_OK;
    }
    if (!aligned(trace, 8) || bytes < (int64_t)plan->sm_count * kTraceWords * 8) return MOE_ERR_INVALID_ARG;
    plan->trace = static_cast<unsigned long long*>(trace);
    return MOE_OK;
}

moe_status_t moe_router_logits(moe_plan_t plan, const uint16_t* x, const uint16_t* W_r,
                               const float* bias, float* logits, void* stream) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    if (plan->T == 0) return MOE_OK;
    if (!x || !W_r || !logits || !aligned(x, 4) || !aligned(W_r, 2) || !aligned(logits, 4) ||
        (bias && !aligned(bias, 4)))
        return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return MOE_ERR_CUDA;
    RouterArgs a;
    a.x = x;
    a.Wr = W_r;
    a.bias = bias;
    a.L = logits;
    a.T = plan->T;
    a.d = plan->d;
    a.E = plan->E;
    a.sm_count = plan->sm_count;
    if (launch_router_logits(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status_t moe_combine(moe_plan_t plan, const void* Y, const float* topk_w, const int32_t* dest,
                         float* out, void* stream) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    if (plan->T == 0) return MOE_OK;
    if (!Y || !topk_w || !dest || !out || !aligned(Y, 16) || !aligned(out, 16) ||
        !aligned(topk_w, 4) || !aligned(dest, 4))
        return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return MOE_ERR_CUDA;
    CombineArgs a;
    a.Y = Y;
    a.y_bf16 = plan->shape.out_dtype == MOE_OUT_BF16 ? 1 : 0;
    a.w = topk_w;
    a.dest = dest;
    a.out = out;
    a.T = plan->T;
    a.k = plan->k;
    a.N = plan->N;
    a.S = (int)plan->S;
    if (launch_combine(a, plan->sm_count, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status_t moe_read_status(const int32_t* dev_status, void* stream, int32_t out[4]) {
    if (!dev_status || !out) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpyAsync(out, dev_status, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return static_cast<moe_status_t>(out[0]);
}

}  // extern "C"
