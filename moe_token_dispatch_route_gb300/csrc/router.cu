// Router logits (the step before the path): L = x @ W_r + bias, computed so that
// routing stays bit-exact against a CPU reference.  The mKernel articles name no
// router; this library fixes its arithmetic as: for each (token, expert), an fp32
// accumulator runs fused multiply-adds over i ascending (a bf16 x bf16 product is
// exact in fp32, so each step is one rounding), then the fp32 bias is added.
//
// CUDA cores, not tensor cores: the tensor cores' internal summation order is not
// specified, and a different order can flip a near-tie in the top-k.  A block
// computes TB tokens x EB experts; each thread owns one expert and 8 tokens (every
// TB/8-th token, so the token groups of one warp read adjacent rows) with 8
// accumulators; 32-wide chunks of x and W_r are staged in shared memory (x rows padded
// to 36 floats, so the float4 reads of adjacent rows fall in different banks).
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRtThreads = 256;
constexpr int kRtChunk = 32;
constexpr int kRtPerThread = 8;
constexpr int kRtStride = kRtChunk + 4;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <int EB>  // experts per block: 8, 16 or 32
__global__ void __launch_bounds__(kRtThreads) router_logits_kernel(const RouterArgs a) {
    constexpr int G = 32 / EB;                                  // token groups per warp
    constexpr int TB = (kRtThreads / 32) * G * kRtPerThread;    // tokens per block
    __shared__ __align__(16) float Xs[TB][kRtStride];
    __shared__ float Ws[kRtChunk][EB];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int eloc = lane % EB;
    const int grp = warp * G + lane / EB;
    const int t0 = blockIdx.x * TB;
    const int e0 = blockIdx.y * EB;
    const int e = e0 + eloc;
    float acc[kRtPerThread];
#pragma unroll
    for (int q = 0; q < kRtPerThread; ++q) acc[q] = 0.f;
    for (int i0 = 0; i0 < a.d; i0 += kRtChunk) {
        for (int idx = tid; idx < TB * kRtChunk; idx += kRtThreads) {
            const int tt = idx / kRtChunk, ii = idx % kRtChunk;
            const int t = t0 + tt;
            Xs[tt][ii] = t < a.T ? bf16_bits_to_float(__ldg(a.x + (size_t)t * a.d + i0 + ii)) : 0.f;
        }
        for (int idx = tid; idx < kRtChunk * EB; idx += kRtThreads) {
            const int ii = idx / EB, ee = idx % EB;
            Ws[ii][ee] = (e0 + ee < a.E) ? bf16_bits_to_float(__ldg(a.Wr + (size_t)(i0 + ii) * a.E + e0 + ee)) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int ii = 0; ii < kRtChunk; ii += 4) {
            const float w0 = Ws[ii][eloc], w1 = Ws[ii + 1][eloc], w2 = Ws[ii + 2][eloc], w3 = Ws[ii + 3][eloc];
#pragma unroll
            for (int q = 0; q < kRtPerThread; ++q) {
                const float4 xv = *reinterpret_cast<const float4*>(&Xs[q * (TB / kRtPerThread) + grp][ii]);
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
        for (int q = 0; q < kRtPerThread; ++q) {
            const int t = t0 + q * (TB / kRtPerThread) + grp;
            if (t < a.T) a.L[(size_t)t * a.E + e] = a.bias ? acc[q] + b : acc[q];
        }
    }
}

template <int EB>
cudaError_t launch_rt(const RouterArgs& a, cudaStream_t stream) {
    constexpr int TB = (kRtThreads / 32) * (32 / EB) * kRtPerThread;
    const dim3 grid((a.T + TB - 1) / TB, (a.E + EB - 1) / EB);
    router_logits_kernel<EB><<<grid, kRtThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits(const RouterArgs& a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    if (a.d % kRtChunk != 0) return cudaErrorInvalidValue;
    if (a.E <= 8) return launch_rt<8>(a, stream);
    if (a.E <= 16) return launch_rt<16>(a, stream);
    return launch_rt<32>(a, stream);
}

}  // namespace moe
