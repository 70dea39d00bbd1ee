// Grouped differential attention prefill with float32 I/O and float32
// arithmetic on the CUDA cores (FFMA).  This is the precision path: every
// product and sum is float32, exp is the accurate expf.
//
// Same operation as the tensor-core prefill ("Differential Attention in
// Large Language Models ...", sections "Differential Attention
// Architecture" and "Headwise Normalization"; noise heads shared by groups of
// signal heads per the "Grouped Differential Attention" abstract).
//
// CTA = (4 RPW query rows, signal head h, batch b), 4 warps with RPW rows
// each (RPW = 4; 1 for dv > 160 or when 16-row CTAs would not fill the GPU).  Keys stream
// through shared memory 32 at a time; lane j scores key j of the tile for
// both maps, the warp keeps both online softmax states of its rows, and lane
// l owns output columns l, l+32, ... of both accumulators.  With one row per
// warp the head width d is a compile-time constant for d = 64 and 128.
#include <cuda_runtime.h>
#include <cstdint>
#include <cmath>

#include "gda.h"
#include "gda_internal.h"

namespace gda {
namespace {

constexpr int kKeys = 32;
constexpr int kThreadsF32 = 128;

struct F32Params {
    const float *q1, *k1, *q2, *k2, *v, *lambda;
    float *out;
    float lambda_init, eps, scale;
    int B, L, hs, hn, d, dv, causal, no_norm;
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// One online-softmax step of one map for one row over a 32-key tile.
// s: this lane's logit (already scaled), -inf if hidden.  Returns this lane's
// weight p; updates (m, l) and returns through alpha the accumulator factor.
__device__ __forceinline__ float online_step(float s, float &m, float &l, float &alpha) {
    const float mt = warp_max(s);
    const float mn = fmaxf(m, mt);
    if (mn == -INFINITY) {   // nothing visible yet
        alpha = 1.f;
        return 0.f;
    }
    alpha = (m == -INFINITY) ? 0.f : expf(m - mn);
    const float p = (s == -INFINITY) ? 0.f : expf(s - mn);
    l = l * alpha + warp_sum(p);
    m = mn;
    return p;
}

template <int NV, int RPW, int DT>   // dv = 32 * NV; RPW rows per warp; DT = d (0: runtime d)
__global__ void __launch_bounds__(kThreadsF32)
gda_prefill_f32_kernel(const F32Params p) {
    extern __shared__ float sm[];
    constexpr int kRows = 4 * RPW;
    const int d = DT ? DT : p.d, dp = d + 1;
    float *q1s = sm;                       // [kRows][d]
    float *q2s = q1s + kRows * d;          // [kRows][d]
    float *k1s = q2s + kRows * d;          // [kKeys][d+1]
    float *k2s = k1s + kKeys * dp;         // [kKeys][d+1]
    float *vs = k2s + kKeys * dp;          // [kKeys][dv]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int q0 = blockIdx.x * kRows;
    const int h = blockIdx.y, b = blockIdx.z;
    const int g = h / (p.hs / p.hn);
    const int dv = p.dv;

    for (int i = threadIdx.x; i < kRows * d; i += blockDim.x) {
        const int r = i / d, e = i % d, qi = q0 + r;
        const bool in = qi < p.L;
        q1s[i] = in ? p.q1[((static_cast<size_t>(b) * p.L + qi) * p.hs + h) * d + e] : 0.f;
        q2s[i] = in ? p.q2[((static_cast<size_t>(b) * p.L + qi) * p.hn + g) * d + e] : 0.f;
    }

    float m1[RPW], l1[RPW], m2[RPW], l2[RPW];
    float o1[RPW][NV], o2[RPW][NV];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        m1[rr] = m2[rr] = -INFINITY;
        l1[rr] = l2[rr] = 0.f;
#pragma unroll
        for (int c = 0; c < NV; ++c) o1[rr][c] = o2[rr][c] = 0.f;
    }

    const int kv_end = p.causal ? min(p.L, q0 + kRows) : p.L;
    for (int k0 = 0; k0 < kv_end; k0 += kKeys) {
        __syncthreads();
        // 16-byte loads, several in flight per thread (d = 64 / 128 and every dv are multiples of 4)
        if constexpr (DT != 0) {
            constexpr int d4 = DT / 4;
#pragma unroll 4
            for (int i = threadIdx.x; i < kKeys * d4; i += blockDim.x) {
                const int j = i / d4, e = (i % d4) * 4, kj = k0 + j;
                float4 x1 = make_float4(0.f, 0.f, 0.f, 0.f), x2 = x1;
                if (kj < p.L) {
                    x1 = *reinterpret_cast<const float4 *>(p.k1 + ((static_cast<size_t>(b) * p.L + kj) * p.hs + h) * d + e);
                    x2 = *reinterpret_cast<const float4 *>(p.k2 + ((static_cast<size_t>(b) * p.L + kj) * p.hn + g) * d + e);
                }
                float *r1 = k1s + j * dp + e, *r2 = k2s + j * dp + e;
                r1[0] = x1.x; r1[1] = x1.y; r1[2] = x1.z; r1[3] = x1.w;
                r2[0] = x2.x; r2[1] = x2.y; r2[2] = x2.z; r2[3] = x2.w;
            }
        } else {
#pragma unroll 4
            for (int i = threadIdx.x; i < kKeys * d; i += blockDim.x) {
                const int j = i / d, e = i % d, kj = k0 + j;
                const bool in = kj < p.L;
                k1s[j * dp + e] = in ? p.k1[((static_cast<size_t>(b) * p.L + kj) * p.hs + h) * d + e] : 0.f;
                k2s[j * dp + e] = in ? p.k2[((static_cast<size_t>(b) * p.L + kj) * p.hn + g) * d + e] : 0.f;
            }
        }
        const int dv4 = dv / 4;
#pragma unroll 4
        for (int i = threadIdx.x; i < kKeys * dv4; i += blockDim.x) {
            const int j = i / dv4, c = (i % dv4) * 4, kj = k0 + j;
            *reinterpret_cast<float4 *>(vs + j * dv + c) =
                kj < p.L ? *reinterpret_cast<const float4 *>(p.v + ((static_cast<size_t>(b) * p.L + kj) * p.hs + h) * dv + c)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();

#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int row = warp * RPW + rr;
            const int qi = q0 + row;
            const int kj = k0 + lane;
            const bool visible = kj < p.L && (!p.causal || kj <= qi);
            float a1 = 0.f, a2 = 0.f;
            const float *q1r = q1s + row * d, *q2r = q2s + row * d;
            const float *k1r = k1s + lane * dp, *k2r = k2s + lane * dp;
#pragma unroll 4
            for (int e = 0; e < d; ++e) {
                a1 = fmaf(q1r[e], k1r[e], a1);
                a2 = fmaf(q2r[e], k2r[e], a2);
            }
            const float s1 = visible ? a1 * p.scale : -INFINITY;
            const float s2 = visible ? a2 * p.scale : -INFINITY;
            float al1, al2;
            const float w1 = online_step(s1, m1[rr], l1[rr], al1);
            const float w2 = online_step(s2, m2[rr], l2[rr], al2);
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                o1[rr][c] *= al1;
                o2[rr][c] *= al2;
            }
            for (int j = 0; j < kKeys; ++j) {
                const float pj1 = __shfl_sync(0xffffffffu, w1, j);
                const float pj2 = __shfl_sync(0xffffffffu, w2, j);
#pragma unroll
                for (int c = 0; c < NV; ++c) {
                    const float vv = vs[j * dv + lane + 32 * c];
                    o1[rr][c] = fmaf(pj1, vv, o1[rr][c]);
                    o2[rr][c] = fmaf(pj2, vv, o2[rr][c]);
                }
            }
        }
    }

    const float lam = p.lambda[h];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int qi = q0 + warp * RPW + rr;
        float o[NV];
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < NV; ++c) {
            o[c] = o1[rr][c] / l1[rr] - lam * (o2[rr][c] / l2[rr]);
            ss = fmaf(o[c], o[c], ss);
        }
        ss = warp_sum(ss);
        const float scale = p.no_norm ? 1.f : (1.f - p.lambda_init) / sqrtf(ss / static_cast<float>(dv) + p.eps);
        if (qi < p.L) {
            float *dst = p.out + ((static_cast<size_t>(b) * p.L + qi) * p.hs + h) * dv;
#pragma unroll
            for (int c = 0; c < NV; ++c) dst[lane + 32 * c] = o[c] * scale;
        }
    }
}

template <int NV, int RPW, int DT>
int launch_nv(const F32Params &p, cudaStream_t stream) {
    constexpr int kRows = 4 * RPW;
    const size_t smem = sizeof(float) * (2 * kRows * p.d + 2 * kKeys * (p.d + 1) + kKeys * p.dv);
    auto kern = gda_prefill_f32_kernel<NV, RPW, DT>;
    if (smem > 48 * 1024) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return record_cuda_error(e);
    }
    dim3 grid((p.L + kRows - 1) / kRows, p.hs, p.B);
    if (grid.y > 65535 || grid.z > 65535) return GDA_ERR_UNSUPPORTED;
    kern<<<grid, kThreadsF32, smem, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

template <int NV>
int launch_rows(const F32Params &p, bool one_row_per_warp, cudaStream_t stream) {
    if (one_row_per_warp) {
        if (p.d == 64) return launch_nv<NV, 1, 64>(p, stream);
        if (p.d == 128) return launch_nv<NV, 1, 128>(p, stream);
        return launch_nv<NV, 1, 0>(p, stream);
    }
    // four rows per warp; one for dv > 160 (more rows' accumulators would spill)
    if constexpr (NV > 5) return launch_nv<NV, 1, 0>(p, stream);
    else return launch_nv<NV, 4, 0>(p, stream);
}

}  // namespace

int launch_prefill_f32(const PrefillArgs &a, cudaStream_t stream) {
    F32Params p;
    p.q1 = static_cast<const float *>(a.q1);
    p.k1 = static_cast<const float *>(a.k1);
    p.q2 = static_cast<const float *>(a.q2);
    p.k2 = static_cast<const float *>(a.k2);
    p.v = static_cast<const float *>(a.v);
    p.lambda = a.lambda;
    p.out = static_cast<float *>(a.out);
    p.lambda_init = a.lambda_init;
    p.eps = a.eps;
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a.d)));
    p.B = a.B;
    p.L = a.L;
    p.hs = a.hs;
    p.hn = a.hn;
    p.d = a.d;
    p.dv = a.dv;
    p.causal = a.causal;
    p.no_norm = (a.flags & GDA_FLAG_NO_NORM) ? 1 : 0;
    // 16-row CTAs unless they would not fill the GPU's SMs: then one row per warp
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    const bool one = static_cast<long long>((a.L + 15) / 16) * a.hs * a.B < sms;
    switch (a.dv / 32) {
        case 1: return launch_rows<1>(p, one, stream);
        case 2: return launch_rows<2>(p, one, stream);
        case 3: return launch_rows<3>(p, one, stream);
        case 4: return launch_rows<4>(p, one, stream);
        case 5: return launch_rows<5>(p, one, stream);
        case 6: return launch_rows<6>(p, one, stream);
        case 7: return launch_rows<7>(p, one, stream);
        case 8: return launch_rows<8>(p, one, stream);
        default: return GDA_ERR_UNSUPPORTED;
    }
}

}  // namespace gda
