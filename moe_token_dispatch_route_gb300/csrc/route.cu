// Routing kernels: top-k over softmax router logits, per-expert histogram,
// exclusive prefix sum and the stable destination permutation.
//
// This is the "route MoE tokens to their expert ranks" half of the
// "MoE Dispatch + GEMM" row in the mKernel articles' table of the five fused
// kernels.  The pages name no routing function; the library reads it as
// softmax top-k with selection on the logits (softmax is monotone), lower
// expert index first between equal logits, gate weight = softmax over all E,
// and a destination order grouped by expert, then token, then slot.
//
// Two launches, no atomics that decide an order:
//  1. route_select_kernel: one CTA per 8-64 tokens (8 warps, or 16 when
//     E > 32), one warp per token at a time.  Each warp holds its token's E logits in registers (E/32 per
//     lane), takes their maximum with a warp max over order-preserving
//     integer keys and their sum of exponentials with xor shuffles, and runs
//     k rounds of a warp arg-max (a warp max of the keys, then a warp min of
//     the expert indices that hold it).  The CTA records which of its tokens picked each
//     expert as a bit mask (one bit per token), from which the per-CTA
//     count and every slot's rank inside the CTA follow by popcount.  The
//     last CTA to finish (ticket counter) turns the per-CTA counts into the
//     global offsets and per-CTA bases (a two-level exclusive scan).
//  2. route_permute_kernel: dest = base[cta][e] + rank; perm[dest] = slot.
//     For T*k <= 8192 the last CTA of the first kernel does this step itself
//     and the second launch is skipped.
#include <algorithm>
#include <climits>
#include <cmath>

#include "route_device.cuh"

namespace moe {
namespace {

template <int VPL, int NT>  // logits per lane: E <= 32 * VPL; NT threads
__global__ void __launch_bounds__(NT) route_select_kernel(const RouteArgs a) {
    extern __shared__ uint32_t smem[];
    select_chunk<VPL, NT>(a, blockIdx.x, smem);
    const int tid = threadIdx.x, E = a.E;
    const int chunk = a.chunk;

    // the last CTA to get here scans the per-CTA counts
    __threadfence();
    __syncthreads();
    __shared__ int s_last;
    if (tid == 0) s_last = (atomicAdd(&a.hdr[kHdrRouteTicket], 1u) == (unsigned)(a.nb - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    __shared__ int part[kMaxE], tot[kMaxE], wsum[NT / 32];
    scan_counts<NT>(a, part, tot, wsum);
    if (a.fuse_permute) {
        // small batches: this CTA also turns every slot's rank into its destination row
        __syncthreads();
        const int S = a.T * a.k;
        for (int s = tid; s < S; s += NT) {
            const int b = (s / a.k) / chunk;
            const int e = __ldcg(a.topk_idx + s);
            if (e < 0 || e >= E) continue;
            const int pos = __ldcg(a.blk + (size_t)b * E + e) + __ldcg(a.dest + s);
            a.dest[s] = pos;
            if (pos >= 0 && pos < S) a.perm[pos] = s;
        }
    }
}

__global__ void __launch_bounds__(256) route_permute_kernel(const RouteArgs a) {
    const long long S = (long long)a.T * a.k;
    for (long long s = (long long)blockIdx.x * blockDim.x + threadIdx.x; s < S;
         s += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(s / a.k);
        const int b = t / a.chunk;
        const int e = a.topk_idx[s];
        if (e < 0 || e >= a.E) continue;
        const int pos = a.blk[(size_t)b * a.E + e] + a.dest[s];
        a.dest[s] = pos;
        if (pos >= 0 && pos < S) a.perm[pos] = (int)s;
    }
}

size_t select_smem_bytes(int E, int k) { return select_smem_words(E, k) * 4; }

template <int VPL>
cudaError_t launch_select(const RouteArgs& a, cudaStream_t stream) {
    constexpr int NT = route_threads(32 * VPL);  // the same for every E of this VPL
    route_select_kernel<VPL, NT><<<a.nb, NT, select_smem_bytes(a.E, a.k), stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t route_prepare_attributes() { return cudaSuccess; }  // < 48 KB dynamic smem

int route_blocks_for(int T, int E, int sm_count) {
    // As many CTAs as keep the last CTA's scan over the [CTAs][E] count table at
    // about 16 loads per thread (one round of loads in flight), and at least one
    // per SM.  A sweep of 8-64 tokens per CTA on one GB300 (graph replays, L2
    // flushed) found the scan's length the limit beyond that: on the
    // Mixtral-shaped batch (8192 tokens, 8 experts) 512 CTAs of 16 tokens route
    // in 13.0 us, 1024 CTAs of 8 in 16.4 us; on the fine-grained one (16384
    // tokens, 64 experts) 2048 CTAs of 8 take 82 us, 256 of 64 take 28 us.
    const int max_blocks = std::max(sm_count, kRouteScanEntries / std::max(1, E));
    int chunk = 8;
    while (chunk < kRouteChunk && (T + chunk - 1) / chunk > max_blocks) chunk *= 2;
    return (T + chunk - 1) / chunk;
}

cudaError_t launch_route(const RouteArgs& args, cudaStream_t stream) {
    // tokens per CTA: the power of two that gives exactly args.nb CTAs
    RouteArgs a = args;
    const int per = (a.T + a.nb - 1) / a.nb;
    a.chunk = 1;
    while (a.chunk < per) a.chunk *= 2;
    if (a.chunk > kRouteChunk || (a.T + a.chunk - 1) / a.chunk != a.nb) return cudaErrorInvalidValue;
    const long long S = (long long)a.T * a.k;
    a.fuse_permute = S <= kRouteFuseSlots ? 1 : 0;
    cudaError_t err;
    if (a.E <= 32) err = launch_select<1>(a, stream);
    else if (a.E <= 64) err = launch_select<2>(a, stream);
    else if (a.E <= 128) err = launch_select<4>(a, stream);
    else if (a.E <= 256) err = launch_select<8>(a, stream);
    else if (a.E <= 512) err = launch_select<16>(a, stream);
    else err = launch_select<32>(a, stream);
    if (err != cudaSuccess || a.fuse_permute) return err;
    const int grid = (int)std::min<long long>((S + 255) / 256, 4096);
    route_permute_kernel<<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
