// moe_route_noalloc: the routing step with its scratch memory in a
// file-scope device array, for callers that cannot allocate device memory.
//
// The routing kernels need scratch beyond their inputs and outputs: one
// int32 count per (routing CTA, expert) and a ticket counter that elects the
// CTA which runs the prefix sum.  moe_route takes that scratch from the
// caller's workspace.  This entry point takes it from g_route_scratch below,
// which every GPU that loads the library holds until the process exits
// (1 MiB + 256 bytes).  The kernels are the same ones moe_route launches.
#include <mutex>

#include "moe.h"
#include "moe_internal.cuh"

namespace moe {
bool plan_route_shape(moe_plan_t plan, int* T, int* E, int* k, int* route_blocks, int* device,
                      int* route_flags);
}

namespace {

constexpr size_t kHeaderInts = 64;          // 256 bytes: the ticket counter lives here
constexpr size_t kTableInts = size_t(1) << 18;  // per-CTA count table: 262144 int32 = 1 MiB
constexpr int kMaxDevices = 64;

// The scratch.  Zero at module load; each call clears the ticket again before
// its launch.  Calls share it, so calls that overlap on the GPU race.
static __device__ __align__(256) int32_t g_route_scratch[kHeaderInts + kTableInts];

// Device address of g_route_scratch, looked up with that device current.  In
// host code the symbol itself is only a host-side stand-in.  Only a successful
// lookup is kept: a failed one (a transient error, or a first call made during a
// stream capture) is retried by the next call on that device.
struct ScratchSlot {
    std::mutex mu;
    void* ptr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];

void* scratch_address(int device) {
    if (device < 0 || device >= kMaxDevices) return nullptr;
    ScratchSlot& s = g_slots[device];
    std::lock_guard<std::mutex> lock(s.mu);
    if (!s.ptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) == cudaSuccess) s.ptr = p;
        else cudaGetLastError();
    }
    return s.ptr;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" moe_status_t moe_route_noalloc(moe_plan_t plan, const float* logits, int32_t* topk_idx,
                                          float* topk_w, int32_t* counts, int32_t* offsets,
                                          int32_t* perm, int32_t* dest, void* stream) {
    int T = 0, E = 0, k = 0, nb = 0, device = 0, flags = 0;
    if (!moe::plan_route_shape(plan, &T, &E, &k, &nb, &device, &flags)) return MOE_ERR_INVALID_ARG;
    if ((size_t)nb * (size_t)E > kTableInts) return MOE_ERR_UNSUPPORTED;  // ceil(T/64)*E > 262144
    if (!counts || !offsets || !aligned4(counts) || !aligned4(offsets)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_idx || !topk_w || !perm || !dest || !aligned4(logits) ||
                  !aligned4(topk_idx) || !aligned4(topk_w) || !aligned4(perm) || !aligned4(dest)))
        return MOE_ERR_INVALID_ARG;

    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return MOE_ERR_CUDA;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
    moe_status_t st = MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* base = scratch_address(device);  // first call on this device: symbol lookup
    if (!base) {
        st = MOE_ERR_CUDA;
    } else if (T == 0) {
        if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess)
            st = MOE_ERR_CUDA;
    } else {
        moe::RouteArgs a;
        a.logits = logits;
        a.topk_idx = topk_idx;
        a.topk_w = topk_w;
        a.counts = counts;
        a.offsets = offsets;
        a.perm = perm;
        a.dest = dest;
        a.hdr = static_cast<uint32_t*>(base);
        a.blk = static_cast<int32_t*>(base) + kHeaderInts;
        a.T = T;
        a.E = E;
        a.k = k;
        a.nb = nb;
        a.sel_bias = nullptr;
        a.renorm = (flags & MOE_ROUTE_RENORM) ? 1 : 0;
        a.sigmoid = (flags & MOE_ROUTE_SIGMOID) ? 1 : 0;
        // the ticket must start at zero; the per-CTA table is fully written before it is read
        if (cudaMemsetAsync(base, 0, kHeaderInts * sizeof(int32_t), s) != cudaSuccess ||
            moe::launch_route(a, s) != cudaSuccess)
            st = MOE_ERR_CUDA;
    }
    if (st != MOE_OK) cudaGetLastError();
    if (prev >= 0 && prev != device) cudaSetDevice(prev);
    return st;
}
