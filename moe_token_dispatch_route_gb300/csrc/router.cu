// Router logits (the step before the path): L = x @ W_r + bias, computed so that
// routing stays bit-exact against a CPU reference.  The mKernel articles name no
// router; this library fixes its arithmetic as: for each (token, expert), an fp32
// accumulator runs fused multiply-adds over i ascending (a bf16 x bf16 product is
// exact in fp32, so each step is one rounding), then the fp32 bias is added.
//
// CUDA cores, not tensor cores: the tensor cores' internal summation order is not
// specified, and a different order can flip a near-tie in the top-k.
//
// Streamed kernel (E a multiple of 8, x and W_r 16-byte aligned): a thread owns one
// token and Q consecutive experts (Q accumulators, each its own chain), a warp 32
// tokens of one group of Q experts, a CTA of 4 warps NGB expert groups x 4/NGB
// rows of 32 tokens.  The reduction runs in 64-element chunks through a 4-stage
// cp.async ring in shared memory: the CTA's x rows (bf16, 136-byte rows, so the 32
// lanes' 8-byte reads from 32 rows take two wavefronts) and W_r's chunk for the
// CTA's experts (bf16, read as warp-wide broadcasts).  Per four reduction elements
// a thread reads 8 bytes of x and four rows of its Q weights and runs 4Q FMAs.
//
// Fallback kernel (any E, 4-byte aligned x): a block computes TB tokens x EB
// experts; each thread owns one expert and P tokens (every TB/P-th token, so the
// token groups of one warp read adjacent rows) with P accumulators, P chosen so the
// grid fills the GPU; the next chunk is loaded into registers while the current
// one is used; 32-wide chunks of x and W_r are staged in shared memory (x rows
// padded to 36 floats, so the float4 reads of adjacent rows fall in different
// banks).
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRtThreads = 256;
constexpr int kRtChunk = 32;
constexpr int kRtStride = kRtChunk + 4;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <int EB, int P>  // experts per block (8, 16 or 32) x tokens per thread (1..8)
__global__ void __launch_bounds__(kRtThreads) router_logits_kernel(const RouterArgs a) {
    constexpr int G = 32 / EB;                    // token groups per warp
    constexpr int TB = (kRtThreads / 32) * G * P; // tokens per block
    constexpr int XPER = TB * kRtChunk / kRtThreads;  // x elements each thread stages per chunk
    constexpr int WPER = (kRtChunk * EB + kRtThreads - 1) / kRtThreads;
    __shared__ __align__(16) float Xs[TB][kRtStride];
    __shared__ float Ws[kRtChunk][EB];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int eloc = lane % EB;
    const int grp = warp * G + lane / EB;
    const int t0 = blockIdx.x * TB;
    const int e0 = blockIdx.y * EB;
    const int e = e0 + eloc;
    float acc[P];
#pragma unroll
    for (int q = 0; q < P; ++q) acc[q] = 0.f;
    // the next chunk is loaded into registers while the current one is used
    uint16_t xr[XPER], wr[WPER];
    auto load_chunk = [&](int i0) {
#pragma unroll
        for (int u = 0; u < XPER; ++u) {
            const int idx = tid + u * kRtThreads;
            const int t = t0 + idx / kRtChunk;
            xr[u] = t < a.T ? __ldg(a.x + (size_t)t * a.d + i0 + idx % kRtChunk) : (uint16_t)0;
        }
#pragma unroll
        for (int u = 0; u < WPER; ++u) {
            const int idx = tid + u * kRtThreads;
            const int ee = idx % EB;
            wr[u] = (idx < kRtChunk * EB && e0 + ee < a.E)
                        ? __ldg(a.Wr + (size_t)(i0 + idx / EB) * a.E + e0 + ee) : (uint16_t)0;
        }
    };
    load_chunk(0);
    for (int i0 = 0; i0 < a.d; i0 += kRtChunk) {
#pragma unroll
        for (int u = 0; u < XPER; ++u) {
            const int idx = tid + u * kRtThreads;
            Xs[idx / kRtChunk][idx % kRtChunk] = bf16_bits_to_float(xr[u]);
        }
#pragma unroll
        for (int u = 0; u < WPER; ++u) {
            const int idx = tid + u * kRtThreads;
            if (idx < kRtChunk * EB) Ws[idx / EB][idx % EB] = bf16_bits_to_float(wr[u]);
        }
        __syncthreads();
        if (i0 + kRtChunk < a.d) load_chunk(i0 + kRtChunk);
#pragma unroll
        for (int ii = 0; ii < kRtChunk; ii += 4) {
            const float w0 = Ws[ii][eloc], w1 = Ws[ii + 1][eloc], w2 = Ws[ii + 2][eloc], w3 = Ws[ii + 3][eloc];
#pragma unroll
            for (int q = 0; q < P; ++q) {
                const float4 xv = *reinterpret_cast<const float4*>(&Xs[q * (TB / P) + grp][ii]);
                acc[q] = fmaf(xv.x, w0, acc[q]);  // i ascending
                acc[q] = fmaf(xv.y, w1, acc[q]);
                acc[q] = fmaf(xv.z, w2, acc[q]);
                acc[q] = fmaf(xv.w, w3, acc[q]);
            }
        }
        __syncthreads();
    }
    if (e < a.E) {
        const float b = a.bias ? __ldg(a.bias + e) : 0.f;
#pragma unroll
        for (int q = 0; q < P; ++q) {
            const int t = t0 + q * (TB / P) + grp;
            if (t < a.T) a.L[(size_t)t * a.E + e] = a.bias ? acc[q] + b : acc[q];
        }
    }
}

constexpr int kRsThreads = 128;
constexpr int kRsCh = 64;                 // reduction elements per stage (d is a multiple of 64)
constexpr int kRsStages = 4;
constexpr int kRsXStride = kRsCh + 4;     // bf16 per staged x row: 136 bytes

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

template <int Q, int NGB>  // experts per thread, expert groups per CTA
constexpr size_t streamed_smem_bytes() {
    return (size_t)kRsStages * (32 * (4 / NGB) * kRsXStride + kRsCh * Q * NGB) * 2;
}

template <int Q, int NGB>
__global__ void __launch_bounds__(kRsThreads) router_logits_streamed(const RouterArgs a) {
    constexpr int TB = 32 * (4 / NGB);             // tokens per CTA
    constexpr int EBLK = Q * NGB;                  // experts per CTA
    constexpr int XST = TB * kRsXStride;           // bf16 per x stage
    constexpr int WST = kRsCh * EBLK;              // bf16 per W stage
    constexpr int XCOPIES = TB * kRsCh / 4;        // 8-byte copies of x per stage
    constexpr int WCOPIES = kRsCh * EBLK / 8;      // 16-byte copies of W per stage
    static_assert(EBLK % 8 == 0, "W rows are copied 8 experts (16 bytes) at a time");
    extern __shared__ __align__(16) uint16_t rs[];
    uint16_t* Xs = rs;                             // [kRsStages][TB][kRsXStride]
    uint16_t* Ws = rs + kRsStages * XST;           // [kRsStages][kRsCh][EBLK]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = warp % NGB;                    // this warp's expert group
    const int tl = (warp / NGB) * 32 + lane;       // this thread's token inside the CTA
    const int t0 = blockIdx.x * TB, e0 = blockIdx.y * EBLK;
    const int nch = a.d / kRsCh;

    auto load_stage = [&](int st, int c) {
        const uint32_t xs = smem_addr(Xs + st * XST), ws = smem_addr(Ws + st * WST);
        for (int j = tid; j < XCOPIES; j += kRsThreads) {
            const int r = j / (kRsCh / 4), part = j % (kRsCh / 4);
            const int t = t0 + r;
            const uint16_t* src = a.x + (t < a.T ? (size_t)t * a.d + (size_t)c * kRsCh + part * 4 : 0);
            cp_async8(xs + (uint32_t)(r * kRsXStride + part * 4) * 2, src, t < a.T ? 8 : 0);
        }
        for (int j = tid; j < WCOPIES; j += kRsThreads) {
            const int i = j / (EBLK / 8), part = j % (EBLK / 8);
            const int e = e0 + part * 8;
            const uint16_t* src = a.Wr + (e < a.E ? (size_t)(c * kRsCh + i) * a.E + e : 0);
            cp_async16_cg_zfill(ws + (uint32_t)(i * EBLK + part * 8) * 2, src, e < a.E ? 16 : 0);
        }
    };

    float acc[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) acc[q] = 0.f;
#pragma unroll
    for (int c = 0; c < kRsStages - 1; ++c) {
        if (c < nch) load_stage(c, c);
        cp_async_commit();
    }
    for (int c = 0; c < nch; ++c) {
        cp_async_wait<kRsStages - 2>();
        __syncthreads();  // chunk c is in; every thread is done with chunk c - 1's stage
        const int cn = c + kRsStages - 1;
        if (cn < nch) load_stage(cn % kRsStages, cn);
        cp_async_commit();
        const uint16_t* xr = Xs + (c % kRsStages) * XST + tl * kRsXStride;
        const uint16_t* wr = Ws + (c % kRsStages) * WST + grp * Q;
#pragma unroll 4
        for (int ii = 0; ii < kRsCh; ii += 4) {
            const uint2 xv = *reinterpret_cast<const uint2*>(xr + ii);
            const float xf[4] = {__uint_as_float(xv.x << 16), __uint_as_float(xv.x & 0xFFFF0000u),
                                 __uint_as_float(xv.y << 16), __uint_as_float(xv.y & 0xFFFF0000u)};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t wv[Q / 2];
                if constexpr (Q == 8) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(wr + (ii + k) * EBLK);
                    wv[0] = w4.x; wv[1] = w4.y; wv[2] = w4.z; wv[3] = w4.w;
                } else {
                    const uint2 w2 = *reinterpret_cast<const uint2*>(wr + (ii + k) * EBLK);
                    wv[0] = w2.x; wv[1] = w2.y;
                }
#pragma unroll
                for (int q = 0; q < Q; ++q) {  // element i = chunk + ii + k: i ascending per accumulator
                    const uint32_t h = wv[q / 2];
                    const float w = __uint_as_float((q & 1) ? (h & 0xFFFF0000u) : (h << 16));
                    acc[q] = fmaf(xf[k], w, acc[q]);
                }
            }
        }
    }
    cp_async_wait<0>();
    const int t = t0 + tl;
    if (t < a.T) {
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int e = e0 + grp * Q + q;
            if (e < a.E) a.L[(size_t)t * a.E + e] = a.bias ? acc[q] + __ldg(a.bias + e) : acc[q];
        }
    }
}

template <int Q, int NGB>
cudaError_t launch_streamed(const RouterArgs& a, cudaStream_t stream) {
    constexpr int TB = 32 * (4 / NGB), EBLK = Q * NGB;
    const dim3 grid((a.T + TB - 1) / TB, (a.E + EBLK - 1) / EBLK);
    router_logits_streamed<Q, NGB><<<grid, kRsThreads, streamed_smem_bytes<Q, NGB>(), stream>>>(a);
    return cudaGetLastError();
}

template <int EB, int P>
cudaError_t launch_rt(const RouterArgs& a, cudaStream_t stream) {
    constexpr int TB = (kRtThreads / 32) * (32 / EB) * P;
    const dim3 grid((a.T + TB - 1) / TB, (a.E + EB - 1) / EB);
    router_logits_kernel<EB, P><<<grid, kRtThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

// tokens per thread: the largest of 8, 4, 2, 1 that still gives at least 2 CTAs per SM
template <int EB>
cudaError_t launch_rt_p(const RouterArgs& a, cudaStream_t stream) {
    const long long eblocks = (a.E + EB - 1) / EB;
    auto ctas = [&](int p) { const int tb = (kRtThreads / 32) * (32 / EB) * p; return eblocks * ((a.T + tb - 1) / tb); };
    const long long want = 2LL * a.sm_count;
    if (ctas(8) >= want) return launch_rt<EB, 8>(a, stream);
    if (ctas(4) >= want) return launch_rt<EB, 4>(a, stream);
    if (ctas(2) >= want) return launch_rt<EB, 2>(a, stream);
    return launch_rt<EB, 1>(a, stream);
}

}  // namespace

cudaError_t launch_router_logits(const RouterArgs& a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    if (a.d % kRtChunk != 0) return cudaErrorInvalidValue;
    const bool streamed = a.E % 8 == 0 && a.d % kRsCh == 0 && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0 &&
                          (reinterpret_cast<uintptr_t>(a.Wr) & 15) == 0;
    if (streamed) {
        // 8 experts per thread for wide routers on large batches, else 4 (more CTAs);
        // expert groups per CTA: 4 when there are that many, else 2
        const int q = (a.E >= 64 && a.T >= 512) ? 8 : 4;
        const int ngb = a.E / q >= 4 ? 4 : 2;
        if (q == 8) return ngb == 4 ? launch_streamed<8, 4>(a, stream) : launch_streamed<8, 2>(a, stream);
        return ngb == 4 ? launch_streamed<4, 4>(a, stream) : launch_streamed<4, 2>(a, stream);
    }
    if (a.E <= 8) return launch_rt_p<8>(a, stream);
    if (a.E <= 16) return launch_rt_p<16>(a, stream);
    return launch_rt_p<32>(a, stream);
}

}  // namespace moe
