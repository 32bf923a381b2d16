// Device code of the routing kernels (route.cu): per-chunk top-k, histogram
// and ranks, and the scan that turns per-chunk counts into offsets and bases.
// Each file that includes it gets its own copy (internal linkage).
#pragma once

#include <climits>
#include <cmath>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr unsigned kRouteFull = 0xFFFFFFFFu;
constexpr int kMaskWords = kRouteChunk / 32;  // bit-mask words per expert

// Order-preserving key of a finite float: a larger float has a larger key,
// equal floats have equal keys (-0.0 is keyed as +0.0), and every key is above
// 0, which stands for "nothing".  key_value inverts it (zeros come back as +0.0).
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Exclusive scan of n <= 1024 ints held in smem `vals`, in place, by NT >= 256
// threads (four values each); returns the total to every thread.  `wsum` is NT/32
// ints of scratch.
template <int NT>
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
        int o = __shfl_up_sync(kRouteFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int pre = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
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
// per-CTA bases blk[b][e] = offsets[e] + sum_{b' < b} count[b'][e].  Shared-memory
// scratch: part and tot of kMaxE ints each, wsum of NT / 32 ints.
template <int NT>
__device__ void scan_counts(const RouteArgs& a, int* part, int* tot, int* wsum) {
    const int tid = threadIdx.x;
    const int E = a.E, nb = a.nb;
    const int G = E >= NT ? 1 : NT / E;  // CTA groups per expert
    // 1. partial sums over contiguous CTA ranges
    for (int job = tid; job < G * E; job += NT) {
        const int e = job % E, g = job / E;
        const int b0 = (int)((long long)nb * g / G), b1 = (int)((long long)nb * (g + 1) / G);
        int s = 0;
        for (int b = b0; b < b1; b += 16) {  // sixteen independent loads in flight
            int v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = b + u < b1 ? __ldcg(a.blk + (size_t)(b + u) * E + e) : 0;
#pragma unroll
            for (int u = 0; u < 16; ++u) s += v[u];
        }
        part[job] = s;
    }
    __syncthreads();
    // 2. per expert: exclusive prefix over the groups, and the total
    for (int e = tid; e < E; e += NT) {
        int run = 0;
        for (int g = 0; g < G; ++g) {
            const int c = part[g * E + e];
            part[g * E + e] = run;
            run += c;
        }
        tot[e] = run;
    }
    __syncthreads();
    for (int e = tid; e < E; e += NT) a.counts[e] = tot[e];
    __syncthreads();
    // 3. exclusive scan over experts -> offsets
    const int total = block_exclusive_scan_1024<NT>(tot, E, wsum);
    for (int e = tid; e < E; e += NT) a.offsets[e] = tot[e];
    if (tid == 0) a.offsets[E] = total;
    // 4. per-CTA bases, written over the per-CTA counts
    for (int job = tid; job < G * E; job += NT) {
        const int e = job % E, g = job / E;
        const int b0 = (int)((long long)nb * g / G), b1 = (int)((long long)nb * (g + 1) / G);
        int run = tot[e] + part[job];
        for (int b = b0; b < b1; b += 16) {
            int v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = b + u < b1 ? __ldcg(a.blk + (size_t)(b + u) * E + e) : 0;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                if (b + u < b1) a.blk[(size_t)(b + u) * E + e] = run;
                run += v[u];
            }
        }
    }
    if (tid == 0) a.hdr[kHdrRouteTicket] = 0;  // ready for the next call
}


// Routing chunk c (tokens [c * chunk, (c + 1) * chunk)) by the calling CTA's NT
// threads: top-k and gates per token (one warp per token at a time), then the
// chunk's per-expert counts into blk[c][*] and every slot's rank among the chunk's
// rows of its expert into dest.  `smem`: E * kMaskWords + kRouteChunk * k words.
template <int VPL, int NT>  // logits per lane: E <= 32 * VPL; NT threads
__device__ void select_chunk(const RouteArgs& a, int c, uint32_t* smem) {
    const int E = a.E, k = a.k;
    uint32_t* mask = smem;                                              // [E][kMaskWords]
    int32_t* sel = reinterpret_cast<int32_t*>(mask + E * kMaskWords);  // [kRouteChunk][k]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < E * kMaskWords; i += NT) mask[i] = 0u;
    __syncthreads();

    const int chunk = a.chunk;
    const int t0 = c * chunk;
    const int ntok = min(chunk, a.T - t0);
    for (int tl = warp; tl < ntok; tl += NT / 32) {
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
        float m = 0.f, s = 0.f;
        if (!a.sigmoid) {
            uint32_t mk = 0u;  // the maximum as a warp max of order keys (exact)
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (live >> i & 1u) mk = max(mk, order_key(v[i]));
            m = key_value(__reduce_max_sync(kRouteFull, mk));
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (live >> i & 1u) s += expf(v[i] - m);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kRouteFull, s, off);
        }
        // selection keys: logit + bias (one fp32 add); the gates still use the logit
        if (a.sel_bias) {
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (live >> i & 1u) v[i] += __ldg(a.sel_bias + lane + 32 * i);
        }

        // k rounds of a warp arg-max on the selection keys: the largest key by a
        // warp max, then the lowest expert index holding it by a warp min
        uint32_t key[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) key[i] = order_key(v[i]);
        int my_e = -1;
        float my_v = 0.f;  // the pick's key value; equal to its logit when there is no bias
        for (int j = 0; j < k; ++j) {
            uint32_t bk = 0u;
            int bi = -1;  // the lane's best live value: its largest key, lowest i between equals
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if ((live >> i & 1u) && key[i] > bk) {
                    bk = key[i];
                    bi = i;
                }
            const uint32_t wk = __reduce_max_sync(kRouteFull, bk);
            const uint32_t we = __reduce_min_sync(
                kRouteFull, (bi >= 0 && bk == wk) ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu);
            if (we != 0xFFFFFFFFu && (int)(we & 31u) == lane) live &= ~(1u << (we >> 5));
            if (lane == j) {
                my_e = we != 0xFFFFFFFFu ? (int)we : -1;
                my_v = key_value(wk);
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
            for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(kRouteFull, ws, off);
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
    int32_t* blk = a.blk + (size_t)c * E;
    for (int e = tid; e < E; e += NT) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kMaskWords; ++w) c += __popc(mask[e * kMaskWords + w]);
        blk[e] = c;
    }
    for (int q = tid; q < ntok * k; q += NT) {
        const int tl = q / k;
        const int e = sel[q];
        if (e < 0 || e >= E) continue;
        const int word = tl >> 5;
        int r = __popc(mask[e * kMaskWords + word] & ((1u << (tl & 31)) - 1u));
        for (int w = 0; w < word; ++w) r += __popc(mask[e * kMaskWords + w]);
        a.dest[(size_t)t0 * k + q] = r;  // rank inside the CTA; made global by the next kernel
    }
}

// shared-memory words select_chunk needs
__host__ __device__ inline size_t select_smem_words(int E, int k) {
    return (size_t)E * kMaskWords + (size_t)kRouteChunk * k;
}

}  // namespace
}  // namespace moe
