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
//  1. route_select_kernel: one CTA per 8-64 tokens, one warp per token at a
//     time.  Each warp holds its token's E logits in registers (E/32 per
//     lane), reduces max and sum-of-exp with xor shuffles and runs k rounds
//     of a warp arg-max.  The CTA records which of its tokens picked each
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

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kMaskWords = kRouteChunk / 32;  // bit-mask words per expert

// (v1, e1) ranks before (v2, e2): larger logit first, lower index between equals.
// Float == treats -0.0 and +0.0 as equal, so the index decides there.
__device__ __forceinline__ bool ranks_before(float v1, int e1, float v2, int e2) {
    return v1 > v2 || (v1 == v2 && e1 < e2);
}

// Exclusive scan of n <= 1024 ints held in smem `vals`, in place, by 256 threads;
// returns the total to every thread.  `wsum` is 8 ints of scratch.
__device__ int block_exclusive_scan_1024(int* vals, int n, int* wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int base = tid * 4;
    int loc[4];
    int sum = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        loc[u] = (base + u < n) ? vals[base + u] : 0;
        sum += loc[u];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int pre = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kRouteThreads / 32; ++w) {
        if (w < warp) pre += wsum[w];
        total += wsum[w];
    }
    int run = pre + incl - sum;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        if (base + u < n) vals[base + u] = run;
        run += loc[u];
    }
    __syncthreads();
    return total;
}

// Runs in the last routing CTA: per-CTA counts blk[b][e] -> counts, offsets and
// per-CTA bases blk[b][e] = offsets[e] + sum_{b' < b} count[b'][e].
__device__ void scan_counts(const RouteArgs& a) {
    __shared__ int part[kMaxE];
    __shared__ int tot[kMaxE];
    __shared__ int wsum[kRouteThreads / 32];
    const int tid = threadIdx.x;
    const int E = a.E, nb = a.nb;
    const int G = E >= kRouteThreads ? 1 : kRouteThreads / E;  // CTA groups per expert
    // 1. partial sums over contiguous CTA ranges
    for (int job = tid; job < G * E; job += kRouteThreads) {
        const int e = job % E, g = job / E;
        const int b0 = (int)((long long)nb * g / G), b1 = (int)((long long)nb * (g + 1) / G);
        int s = 0;
        int b = b0;
        for (; b + 8 <= b1; b += 8) {  // eight independent loads in flight
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(a.blk + (size_t)(b + u) * E + e);
#pragma unroll
            for (int u = 0; u < 8; ++u) s += v[u];
        }
        for (; b < b1; ++b) s += __ldcg(a.blk + (size_t)b * E + e);
        part[job] = s;
    }
    __syncthreads();
    // 2. per expert: exclusive prefix over the groups, and the total
    for (int e = tid; e < E; e += kRouteThreads) {
        int run = 0;
        for (int g = 0; g < G; ++g) {
            const int c = part[g * E + e];
            part[g * E + e] = run;
            run += c;
        }
        tot[e] = run;
    }
    __syncthreads();
    for (int e = tid; e < E; e += kRouteThreads) a.counts[e] = tot[e];
    __syncthreads();
    // 3. exclusive scan over experts -> offsets
    const int total = block_exclusive_scan_1024(tot, E, wsum);
    for (int e = tid; e < E; e += kRouteThreads) a.offsets[e] = tot[e];
    if (tid == 0) a.offsets[E] = total;
    // 4. per-CTA bases, written over the per-CTA counts
    for (int job = tid; job < G * E; job += kRouteThreads) {
        const int e = job % E, g = job / E;
        const int b0 = (int)((long long)nb * g / G), b1 = (int)((long long)nb * (g + 1) / G);
        int run = tot[e] + part[job];
        int b = b0;
        for (; b + 8 <= b1; b += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(a.blk + (size_t)(b + u) * E + e);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                a.blk[(size_t)(b + u) * E + e] = run;
                run += v[u];
            }
        }
        for (; b < b1; ++b) {
            int* p = a.blk + (size_t)b * E + e;
            const int c = __ldcg(p);
            *p = run;
            run += c;
        }
    }
    if (tid == 0) a.hdr[kHdrRouteTicket] = 0;  // ready for the next call
}

template <int VPL>  // logits per lane: E <= 32 * VPL
__global__ void __launch_bounds__(kRouteThreads) route_select_kernel(const RouteArgs a) {
    extern __shared__ uint32_t smem[];
    const int E = a.E, k = a.k;
    uint32_t* mask = smem;                                              // [E][kMaskWords]
    int32_t* sel = reinterpret_cast<int32_t*>(mask + E * kMaskWords);  // [kRouteChunk][k]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < E * kMaskWords; i += kRouteThreads) mask[i] = 0u;
    __syncthreads();

    const int chunk = a.chunk;
    const int t0 = blockIdx.x * chunk;
    const int ntok = min(chunk, a.T - t0);
    for (int tl = warp; tl < ntok; tl += kRouteThreads / 32) {
        const int t = t0 + tl;
        const float* L = a.logits + (size_t)t * E;
        float v[VPL];
        uint32_t live = 0;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                v[i] = __ldg(L + e);
                live |= 1u << i;
            } else {
                v[i] = 0.f;
            }
        }
        // softmax statistics over all E logits (unused by the logistic score)
        float m = -INFINITY, s = 0.f;
        if (!a.sigmoid) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (live >> i & 1u) m = fmaxf(m, v[i]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (live >> i & 1u) s += expf(v[i] - m);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
        }
        // selection keys: logit + bias (one fp32 add); the gates still use the logit
        if (a.sel_bias) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (live >> i & 1u) v[i] += __ldg(a.sel_bias + lane + 32 * i);
        }

        int my_e = -1;
        float my_v = 0.f;  // the pick's key; equal to its logit when there is no bias
        for (int j = 0; j < k; ++j) {
            float bv = 0.f;
            int be = INT_MAX;  // INT_MAX: nothing left in this lane
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                if (live >> i & 1u) {
                    if (be == INT_MAX || v[i] > bv) {  // strict: lower index kept between equals
                        bv = v[i];
                        be = lane + 32 * i;
                    }
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(kFull, bv, off);
                const int oe = __shfl_xor_sync(kFull, be, off);
                if (oe != INT_MAX && (be == INT_MAX || ranks_before(ov, oe, bv, be))) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane) live &= ~(1u << (be >> 5));
            if (lane == j) {
                my_e = be;
                my_v = bv;
            }
        }
        float my_w = 0.f;
        if (lane < k) {
            const float lg = a.sel_bias ? __ldg(L + my_e) : my_v;
            my_w = a.sigmoid ? 1.f / (1.f + expf(-lg)) : expf(lg - m) / s;
        }
        if (a.renorm) {  // divide by the sum of the token's k gates
            float ws = my_w;  // 0 in lanes >= k
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(kFull, ws, off);
            my_w = my_w / ws;
        }
        if (lane < k) {
            a.topk_idx[(size_t)t * k + lane] = my_e;
            a.topk_w[(size_t)t * k + lane] = my_w;
            sel[tl * k + lane] = my_e;
            if (my_e >= 0 && my_e < E)  // always true for k <= E; guards the shared-memory index
                atomicOr(&mask[my_e * kMaskWords + (tl >> 5)], 1u << (tl & 31));
        }
    }
    __syncthreads();

    // per-CTA counts and each slot's rank among this CTA's rows of its expert
    int32_t* blk = a.blk + (size_t)blockIdx.x * E;
    for (int e = tid; e < E; e += kRouteThreads) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kMaskWords; ++w) c += __popc(mask[e * kMaskWords + w]);
        blk[e] = c;
    }
    for (int q = tid; q < ntok * k; q += kRouteThreads) {
        const int tl = q / k;
        const int e = sel[q];
        if (e < 0 || e >= E) continue;
        const int word = tl >> 5;
        int r = __popc(mask[e * kMaskWords + word] & ((1u << (tl & 31)) - 1u));
        for (int w = 0; w < word; ++w) r += __popc(mask[e * kMaskWords + w]);
        a.dest[(size_t)t0 * k + q] = r;  // rank inside the CTA; made global by the next kernel
    }

    // the last CTA to get here scans the per-CTA counts
    __threadfence();
    __syncthreads();
    __shared__ int s_last;
    if (tid == 0) s_last = (atomicAdd(&a.hdr[kHdrRouteTicket], 1u) == (unsigned)(a.nb - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    scan_counts(a);
    if (a.fuse_permute) {
        // small batches: this CTA also turns every slot's rank into its destination row
        __syncthreads();
        const int S = a.T * a.k;
        for (int s = tid; s < S; s += kRouteThreads) {
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

size_t select_smem_bytes(int E, int k) {
    return (size_t)E * kMaskWords * 4 + (size_t)kRouteChunk * k * 4;
}

template <int VPL>
cudaError_t launch_select(const RouteArgs& a, cudaStream_t stream) {
    route_select_kernel<VPL><<<a.nb, kRouteThreads, select_smem_bytes(a.E, a.k), stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t route_prepare_attributes() { return cudaSuccess; }  // < 48 KB dynamic smem

int route_blocks_for(int T, int E, int sm_count) {
    // As many CTAs as keep the last CTA's scan over the [CTAs][E] count table near
    // 64 loads per thread, and at least one per SM: with few experts that means one
    // token per warp (no serial token loop), with many a few tokens per warp.
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
