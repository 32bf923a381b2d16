// Router logits (the step before the path): L = x @ W_r + bias, computed so that
// routing stays bit-exact against a CPU reference.  The mKernel articles name no
// router; this library fixes its arithmetic as: for each (token, expert), an fp32
// accumulator runs fused multiply-adds over i ascending (a bf16 x bf16 product is
// exact in fp32, so each step is one rounding), then the fp32 bias is added.
//
// CUDA cores, not tensor cores: the tensor cores' internal summation order is not
// specified, and a different order can flip a near-tie in the top-k.  A block
// computes TB tokens x EB experts; each thread owns one expert and P tokens (every
// TB/P-th token, so the token groups of one warp read adjacent rows) with P
// accumulators, P chosen so the grid fills the GPU; the next chunk is loaded into
// registers while the current one is used; 32-wide chunks of x and W_r are staged in shared memory (x rows padded
// to 36 floats, so the float4 reads of adjacent rows fall in different banks).
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
    if (a.E <= 8) return launch_rt_p<8>(a, stream);
    if (a.E <= 16) return launch_rt_p<16>(a, stream);
    return launch_rt_p<32>(a, stream);
}

}  // namespace moe
