// Router logits (the step before the path): L = x @ W_r + bias, computed so that
// routing stays bit-exact against a CPU reference.  The mKernel articles name no
// router; this library fixes its arithmetic as: for each (token, expert), an fp32
// accumulator runs fused multiply-adds over i ascending (a bf16 x bf16 product is
// exact in fp32, so each step is one rounding), then the fp32 bias is added.
//
// CUDA cores, not tensor cores: the tensor cores' internal summation order is not
// specified, and a different order can flip a near-tie in the top-k.
//
// Streamed kernel (E a multiple of 8, d of 64, x and W_r 16-byte aligned): a
// thread owns P tokens and Q consecutive experts (P x Q accumulators, each its own
// chain), a warp 32 token rows of one group of Q experts, a CTA NGB expert groups x
// WPG warp rows.  The reduction runs in CH-element chunks through a 4-stage
// cp.async ring in shared memory holding the CTA's x rows (bf16, rows padded by 8
// bytes, so the 32 lanes' 8-byte reads from 32 rows take two wavefronts) and W_r's
// chunk for the CTA's experts; each chunk of W_r is widened to fp32 once per CTA
// and then read as warp-wide broadcasts.  The chunk loop is unrolled whole, so
// shared-memory loads run ahead of the FMA chains.  Two shapes:
//   wide   (P 2, Q 8, 128 tokens x 32 experts per CTA of 8 warps, CH 64), once its
//          grid covers every SM: one fp32 weight read feeds 16 FMAs, so shared-memory
//          wavefronts stay below the FMA issue rate;
//   narrow (P 1, Q 2, 32 tokens x 8 experts per CTA of 4 warps, CH 128): small
//          batches and few experts, where the work is a few warps per SM and the
//          time goes to the chains' latency and the per-chunk barriers.
//
// Fallback kernel (any E, d a multiple of 16, 4-byte aligned x): a block computes TB tokens x EB
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
            const int i = i0 + idx % kRtChunk;
            xr[u] = (t < a.T && i < a.d) ? __ldg(a.x + (size_t)t * a.d + i) : (uint16_t)0;
        }
#pragma unroll
        for (int u = 0; u < WPER; ++u) {
            const int idx = tid + u * kRtThreads;
            const int ee = idx % EB;
            wr[u] = (idx < kRtChunk * EB && e0 + ee < a.E && i0 + idx / EB < a.d)
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
            if (i0 + ii >= a.d) break;  // a last chunk of 16 (d % 32 == 16): no step past d
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

constexpr int kRsStages = 4;

__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Streamed-kernel shape: Q experts x P tokens per thread, NGB expert groups and
// WPG warp rows per CTA, CH reduction elements per ring stage.
template <int Q_, int P_, int NGB_, int WPG_, int CH_>
struct RsCfg {
    static constexpr int Q = Q_, P = P_, NGB = NGB_, WPG = WPG_, CH = CH_;
    static constexpr int kThreads = 32 * NGB * WPG;
    static constexpr int TB = 32 * WPG * P;      // tokens per CTA
    static constexpr int EBLK = Q * NGB;         // experts per CTA
    static constexpr int XS = CH + 4;            // bf16 per staged x row (2 * CH + 8 bytes)
    static constexpr int XST = TB * XS;          // bf16 per x stage
    static constexpr int WST = CH * EBLK;        // bf16 per W stage
    static constexpr size_t kSmem = (size_t)kRsStages * (XST + WST) * 2 + (size_t)WST * 4;
    static_assert(EBLK % 8 == 0, "W rows are copied 8 experts (16 bytes) at a time");
    static_assert(Q == 2 || Q % 4 == 0, "a thread's Q weights are read as float2 or float4 words");
    static_assert(CH % 4 == 0, "x is read four elements at a time");
};

// Q consecutive fp32 weights of one reduction element
template <int Q>
__device__ __forceinline__ void weights_f32(const float* p, float (&w)[Q]) {
    if constexpr (Q == 2) {
        const float2 v = *reinterpret_cast<const float2*>(p);
        w[0] = v.x; w[1] = v.y;
    } else {
#pragma unroll
        for (int u = 0; u < Q / 4; ++u) {
            const float4 v = *reinterpret_cast<const float4*>(p + 4 * u);
            w[4 * u] = v.x; w[4 * u + 1] = v.y; w[4 * u + 2] = v.z; w[4 * u + 3] = v.w;
        }
    }
}

template <class C>
__global__ void __launch_bounds__(C::kThreads) router_logits_streamed(const RouterArgs a) {
    constexpr int Q = C::Q, P = C::P, NGB = C::NGB, WPG = C::WPG, CH = C::CH;
    constexpr int NT = C::kThreads, TB = C::TB, EBLK = C::EBLK, XS = C::XS, XST = C::XST, WST = C::WST;
    constexpr int XCOPIES = TB * CH / 4;           // 8-byte copies of x per stage
    constexpr int WCOPIES = WST / 8;               // 16-byte copies of W per stage
    extern __shared__ __align__(16) uint16_t rs[];
    uint16_t* Xs = rs;                             // [kRsStages][TB][XS]
    uint16_t* Ws = rs + kRsStages * XST;           // [kRsStages][CH][EBLK]
    float* Wf = reinterpret_cast<float*>(Ws + kRsStages * WST);  // [CH][EBLK], the current chunk
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = warp % NGB;                    // this warp's expert group
    const int tl = (warp / NGB) * 32 + lane;       // this thread's first token inside the CTA
    const int t0 = blockIdx.x * TB, e0 = blockIdx.y * EBLK;
    const int nch = a.d / CH;

    auto load_stage = [&](int st, int c) {
        const uint32_t xs = smem_addr(Xs + st * XST), ws = smem_addr(Ws + st * WST);
        for (int j = tid; j < XCOPIES; j += NT) {
            const int r = j / (CH / 4), part = j % (CH / 4);
            const int t = t0 + r;
            const uint16_t* src = a.x + (t < a.T ? (size_t)t * a.d + (size_t)c * CH + part * 4 : 0);
            cp_async8(xs + (uint32_t)(r * XS + part * 4) * 2, src, t < a.T ? 8 : 0);
        }
        for (int j = tid; j < WCOPIES; j += NT) {
            const int i = j / (EBLK / 8), part = j % (EBLK / 8);
            const int e = e0 + part * 8;
            const uint16_t* src = a.Wr + (e < a.E ? (size_t)(c * CH + i) * a.E + e : 0);
            cp_async16_cg_zfill(ws + (uint32_t)(i * EBLK + part * 8) * 2, src, e < a.E ? 16 : 0);
        }
    };

    float acc[P][Q];
#pragma unroll
    for (int p = 0; p < P; ++p)
#pragma unroll
        for (int q = 0; q < Q; ++q) acc[p][q] = 0.f;
#pragma unroll
    for (int c = 0; c < kRsStages - 1; ++c) {
        if (c < nch) load_stage(c, c);
        cp_async_commit();
    }
    for (int c = 0; c < nch; ++c) {
        cp_async_wait<kRsStages - 2>();
        __syncthreads();  // chunk c is in; every thread is done with chunk c - 1 (and Wf)
        const int cn = c + kRsStages - 1;
        if (cn < nch) load_stage(cn % kRsStages, cn);
        cp_async_commit();
        {  // widen the chunk's weights once; each is used by the CTA's TB tokens
            const uint4* src = reinterpret_cast<const uint4*>(Ws + (c % kRsStages) * WST);
            float4* dst = reinterpret_cast<float4*>(Wf);
            for (int j = tid; j < WST / 8; j += NT) {
                const uint4 v = src[j];
                dst[2 * j] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                                         __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
                dst[2 * j + 1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                                             __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
            }
        }
        __syncthreads();
        const uint16_t* xr = Xs + (c % kRsStages) * XST + tl * XS;
        const float* wr = Wf + grp * Q;
#pragma unroll
        for (int ii = 0; ii < CH; ii += 4) {  // unrolled whole, so the loads run ahead of the FMAs
            float xf[P][4];
#pragma unroll
            for (int p = 0; p < P; ++p) {  // token p of this thread: row tl + 32 * WPG * p
                const uint2 xv = *reinterpret_cast<const uint2*>(xr + p * 32 * WPG * XS + ii);
                xf[p][0] = __uint_as_float(xv.x << 16);
                xf[p][1] = __uint_as_float(xv.x & 0xFFFF0000u);
                xf[p][2] = __uint_as_float(xv.y << 16);
                xf[p][3] = __uint_as_float(xv.y & 0xFFFF0000u);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float w[Q];
                weights_f32<Q>(wr + (ii + k) * EBLK, w);
#pragma unroll
                for (int p = 0; p < P; ++p)
#pragma unroll
                    for (int q = 0; q < Q; ++q)  // element i = chunk + ii + k: i ascending per accumulator
                        acc[p][q] = fmaf(xf[p][k], w[q], acc[p][q]);
            }
        }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int t = t0 + tl + 32 * WPG * p;
        if (t >= a.T) continue;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int e = e0 + grp * Q + q;
            if (e < a.E) a.L[(size_t)t * a.E + e] = a.bias ? acc[p][q] + __ldg(a.bias + e) : acc[p][q];
        }
    }
}

template <class C>
cudaError_t streamed_attributes() {
    if (C::kSmem <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(router_logits_streamed<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)C::kSmem);
}

template <class C>
cudaError_t launch_streamed(const RouterArgs& a, cudaStream_t stream) {
    const dim3 grid((a.T + C::TB - 1) / C::TB, (a.E + C::EBLK - 1) / C::EBLK);
    router_logits_streamed<C><<<grid, C::kThreads, C::kSmem, stream>>>(a);
    return cudaGetLastError();
}

// The streamed shapes.  Wide: 8 experts x 2 tokens per thread, 128 tokens x 32
// experts per CTA of 8 warps (each weight read from shared memory feeds 16 FMAs).
// Narrow: 2 experts x 1 token per thread, 32 tokens x 8 experts per CTA of 4 warps,
// 128-element stages (more and shorter chains, for small batches and few experts).
using RsWide = RsCfg<8, 2, 4, 2, 64>;
using RsNarrow = RsCfg<2, 1, 4, 1, 128>;
using RsNarrow64 = RsCfg<2, 1, 4, 1, 64>;  // d not a multiple of 128

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

cudaError_t router_prepare_attributes() {
    cudaError_t e = streamed_attributes<RsWide>();
    if (e == cudaSuccess) e = streamed_attributes<RsNarrow>();
    if (e == cudaSuccess) e = streamed_attributes<RsNarrow64>();
    return e;
}

cudaError_t launch_router_logits(const RouterArgs& a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    if (a.d % 16 != 0) return cudaErrorInvalidValue;
    const bool streamed = a.E % 8 == 0 && a.d % 64 == 0 && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0 &&
                          (reinterpret_cast<uintptr_t>(a.Wr) & 15) == 0;
    if (streamed) {
        // the wide shape once its grid covers every SM, else the narrow one
        const long long wide_ctas = (long long)((a.T + RsWide::TB - 1) / RsWide::TB) *
                                    ((a.E + RsWide::EBLK - 1) / RsWide::EBLK);
        if (a.E >= RsWide::EBLK && wide_ctas >= a.sm_count) return launch_streamed<RsWide>(a, stream);
        if (a.d % RsNarrow::CH == 0) return launch_streamed<RsNarrow>(a, stream);
        return launch_streamed<RsNarrow64>(a, stream);
    }
    if (a.E <= 8) return launch_rt_p<8>(a, stream);
    if (a.E <= 16) return launch_rt_p<16>(a, stream);
    return launch_rt_p<32>(a, stream);
}

}  // namespace moe
