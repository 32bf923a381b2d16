// Combine: the step after "MoE Dispatch + GEMM" (the mKernel articles' table of
// the five fused kernels describes only the dispatch side).  It undoes the
// destination permutation and weights each token's k expert outputs by its gates:
//   out[t][n] = sum_{j<k} w[t*k+j] * Y[dest[t*k+j]][n]
// in fp32 with fused multiply-adds in ascending j, so the result is the same on
// every run.  HBM-bound: it reads T*k rows of Y (gathered; fp32 or bf16, whose
// values are exactly representable in fp32) and writes T rows.
//
// One CTA per (token, block of 1024 columns); each thread owns 4 consecutive
// columns and, for k <= 8, keeps its k gathered loads in flight at once.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kCombineCols = kCombineThreads * 4;

// Four consecutive columns of Y row `row`, widened to fp32 (a bf16 value is exact in fp32).
__device__ __forceinline__ float4 load_y4(const CombineArgs& a, int row, int n) {
    if (a.y_bf16) {
        const uint2 h = __ldcs(reinterpret_cast<const uint2*>(
            static_cast<const uint16_t*>(a.Y) + (size_t)row * a.N + n));
        return make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xFFFF0000u),
                           __uint_as_float(h.y << 16), __uint_as_float(h.y & 0xFFFF0000u));
    }
    return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(a.Y) + (size_t)row * a.N + n));
}

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& y) {
    acc.x = fmaf(w, y.x, acc.x);
    acc.y = fmaf(w, y.y, acc.y);
    acc.z = fmaf(w, y.z, acc.z);
    acc.w = fmaf(w, y.w, acc.w);
}

// KMAX > 0 (k <= KMAX): all of a token's destinations and gates are read, then all its
// rows are loaded, then summed, so a thread has k row loads in flight at once.  KMAX = 0
// (any k): one slot at a time.  Both sum in ascending j and skip the same slots, so the
// bits do not depend on which one runs.  Each k bound is its own kernel: the KMAX = 8
// registers would cut the occupancy of a k = 2 launch.
template <int KMAX>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
    const int nblk = (a.N + kCombineCols - 1) / kCombineCols;
    const long long total = (long long)a.T * nblk;
    for (long long b = blockIdx.x; b < total; b += gridDim.x) {
        const int t = (int)(b / nblk);
        const int n = (int)(b % nblk) * kCombineCols + threadIdx.x * 4;
        if (n >= a.N) continue;  // N % 16 == 0, so n < N implies n + 3 < N
        const long long s0 = (long long)t * a.k;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (KMAX > 0) {
            int row[KMAX];
            float wj[KMAX];
            float4 y[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                const bool live = j < a.k;
                row[j] = live ? __ldg(a.dest + s0 + j) : -1;
                wj[j] = live ? __ldg(a.w + s0 + j) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (row[j] >= 0 && row[j] < a.S) y[j] = load_y4(a, row[j], n);
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (row[j] >= 0 && row[j] < a.S) fma4(acc, wj[j], y[j]);
        } else {
            for (int j = 0; j < a.k; ++j) {
                const int row = __ldg(a.dest + s0 + j);
                if (row < 0 || row >= a.S) continue;
                fma4(acc, __ldg(a.w + s0 + j), load_y4(a, row, n));
            }
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
    if (a.k <= 2) combine_kernel<2><<<grid, kCombineThreads, 0, stream>>>(a);
    else if (a.k <= 4) combine_kernel<4><<<grid, kCombineThreads, 0, stream>>>(a);
    else if (a.k <= 8) combine_kernel<8><<<grid, kCombineThreads, 0, stream>>>(a);
    else combine_kernel<0><<<grid, kCombineThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
