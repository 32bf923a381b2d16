// Combine: the step after "MoE Dispatch + GEMM" (the mKernel articles' table of
// the five fused kernels describes only the dispatch side).  It undoes the
// destination permutation and weights each token's k expert outputs by its gates:
//   out[t][n] = sum_{j<k} w[t*k+j] * Y[dest[t*k+j]][n]
// in fp32 with fused multiply-adds in ascending j, so the result is the same on
// every run.  HBM-bound: it reads T*k rows of Y (gathered; fp32 or bf16, whose
// values are exactly representable in fp32) and writes T rows.
//
// One CTA per (token, block of 1024 columns); each thread owns 4 consecutive
// columns and keeps its k gathered 16-byte loads in flight.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kCombineCols = kCombineThreads * 4;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
    const int nblk = (a.N + kCombineCols - 1) / kCombineCols;
    const long long total = (long long)a.T * nblk;
    for (long long b = blockIdx.x; b < total; b += gridDim.x) {
        const int t = (int)(b / nblk);
        const int n = (int)(b % nblk) * kCombineCols + threadIdx.x * 4;
        if (n >= a.N) continue;  // N % 16 == 0, so n < N implies n + 3 < N
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < a.k; ++j) {
            const long long s = (long long)t * a.k + j;
            const int row = __ldg(a.dest + s);
            if (row < 0 || row >= a.S) continue;
            const float wj = __ldg(a.w + s);
            float4 y;
            if (a.y_bf16) {
                const uint2 h = __ldcs(reinterpret_cast<const uint2*>(
                    static_cast<const uint16_t*>(a.Y) + (size_t)row * a.N + n));
                y = make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xFFFF0000u),
                                __uint_as_float(h.y << 16), __uint_as_float(h.y & 0xFFFF0000u));
            } else {
                y = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(a.Y) + (size_t)row * a.N + n));
            }
            acc.x = fmaf(wj, y.x, acc.x);
            acc.y = fmaf(wj, y.y, acc.y);
            acc.z = fmaf(wj, y.z, acc.z);
            acc.w = fmaf(wj, y.w, acc.w);
        }
        __stcs(reinterpret_cast<float4*>(a.out + (size_t)t * a.N + n), acc);
    }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int sm_count, cudaStream_t stream) {
    const int nblk = (a.N + kCombineCols - 1) / kCombineCols;
    const long long total = (long long)a.T * nblk;
    const int grid = (int)std::min<long long>(total, (long long)sm_count * 8);
    if (grid <= 0) return cudaSuccess;
    combine_kernel<<<grid, kCombineThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
