// Gradients of grouped differential attention, float32 on the CUDA cores.
//
// Forward, per batch b, signal head h (noise head g = h / r) and query row i
// ("Differential Attention in Large Language Models ...", sections
// "Differential Attention Architecture" and "Headwise Normalization"; noise
// heads shared by groups per the "Grouped Differential Attention" abstract):
//   a1 = softmax(s1), s1_j = q1_i . k1_j / sqrt d;  a2 = softmax(s2) (noise head g)
//   O1 = sum_j a1_j v_j,  O2 = sum_j a2_j v_j,  o = O1 - lambda_h O2
//   y = (1 - lambda_init) o / rms,  rms = sqrt(mean(o^2) + eps)
// Backward of sum(dy . y), by the chain rule:
//   do   = (c / rms) (dy - o (dy . o) / (dv rms^2)),  c = 1 - lambda_init   (do = dy without the norm)
//   dA_ij = do_i . v_j,  D1_i = do_i . O1_i,  D2_i = do_i . O2_i
//   ds1_ij = a1_ij (dA_ij - D1_i),  ds2_ij = -lambda_h a2_ij (dA_ij - D2_i)
//   dq1_i = sum_j ds1_ij k1_j / sqrt d,   dk1_j = sum_i ds1_ij q1_i / sqrt d
//   dq2_{g,i} = sum_{h in g} sum_j ds2_ij k2_j / sqrt d,  dk2_{g,j} likewise with q2_i
//   dv_j = sum_i (a1_ij - lambda_h a2_ij) do_i,   dlambda_h = -sum_{b,i} D2_i
//
// Three kernels:
//   row pass    (CTA = 16 query rows of one (b, h), 2 per warp): the forward's online
//               softmax gives the row statistics and O1, O2; then do, D1, D2
//               and a second sweep over the keys accumulates dq1 and this
//               head's share of dq2.  Row statistics and do go to the workspace.
//   column pass (CTA = 16 keys of one (b, h), 2 per warp): sweeps the query rows that see
//               its keys, recomputes a1, a2 from the row statistics and
//               accumulates dv, dk1 and this head's share of dk2.
//   reduce      sums the shares of each noise head's group and the rows'
//               dlambda terms (fixed order: results do not depend on timing).
#include <cuda_runtime.h>
#include <cstdint>
#include <cmath>

#include "gda.h"
#include "gda_internal.h"

namespace gda {
namespace {

constexpr int kBRows = 32;       // query rows (row pass) or keys (column pass) per CTA
constexpr int kBTile = 32;       // keys (row pass) or query rows (column pass) per shared-memory tile
constexpr int kBThreads = 256;   // 8 warps
constexpr int kRPW = kBRows / (kBThreads / 32);   // rows (keys) per warp

struct BwdParams {
    const float *q1, *k1, *q2, *k2, *v, *lambda, *dy;
    float *dq1, *dk1, *dq2, *dk2, *dvo, *dlambda;
    // workspace
    float *stats;     // [B, L, hs, 6]: m1, l1, m2, l2, D1, D2
    float *dO;        // [B, L, hs, dv]
    float *dq2h;      // [B, L, hs, d]: each signal head's share of dq2
    float *dk2h;      // [B, L, hs, d]
    float *dlam_row;  // [B, L, hs]
    float lambda_init, eps, scale;
    int B, L, hs, hn, d, dv, causal, no_norm;
};

__device__ __forceinline__ float warp_max_b(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum_b(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ size_t rix(const BwdParams &p, int b, int i, int h) {
    return (static_cast<size_t>(b) * p.L + i) * p.hs + h;
}

// Shared-memory rows read one per lane are padded by 4 floats (16-byte
// aligned float4 reads, at most the 4 wavefronts 512 bytes need); rows read
// by the whole warp at once (broadcast) are not padded.  Each warp's rows
// (keys) share every load: the row loops sit inside the load loops.

template <int D>
__device__ __forceinline__ float4 ld4(const float *base, int i) {
    return reinterpret_cast<const float4 *>(base)[i];
}

__device__ __forceinline__ float dot4(const float4 &a, const float4 &b, float acc) {
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}

// -------------------------------------------------------------- row pass --
template <int ND, int NV>   // d = 32 ND, dv = 32 NV
__global__ void __launch_bounds__(kBThreads)
gda_bwd_row_kernel(const BwdParams p) {
    extern __shared__ float sm[];
    constexpr int d = 32 * ND, dv = 32 * NV, dk = d + 4, dvk = dv + 4;
    float *q1s = sm;                       // [kBRows][d]      broadcast rows
    float *q2s = q1s + kBRows * d;         // [kBRows][d]
    float *k1s = q2s + kBRows * d;         // [kBTile][d+4]    one row per lane
    float *k2s = k1s + kBTile * dk;        // [kBTile][d+4]
    float *vs = k2s + kBTile * dk;         // [kBTile][dv+4]
    float *dos = vs + kBTile * dvk;        // [kBRows][dv]     broadcast rows

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int q0 = blockIdx.x * kBRows;
    const int h = blockIdx.y, b = blockIdx.z;
    const int g = h / (p.hs / p.hn);
    const float lam = p.lambda[h];

    for (int t = threadIdx.x; t < kBRows * d / 4; t += blockDim.x) {
        const int r = t / (d / 4), e = (t % (d / 4)) * 4, qi = q0 + r;
        float4 x1 = make_float4(0.f, 0.f, 0.f, 0.f), x2 = x1;
        if (qi < p.L) {
            x1 = *reinterpret_cast<const float4 *>(p.q1 + rix(p, b, qi, h) * d + e);
            x2 = *reinterpret_cast<const float4 *>(p.q2 + ((static_cast<size_t>(b) * p.L + qi) * p.hn + g) * d + e);
        }
        *reinterpret_cast<float4 *>(q1s + r * d + e) = x1;
        *reinterpret_cast<float4 *>(q2s + r * d + e) = x2;
    }

    auto load_keys = [&](int k0) {
        __syncthreads();
#pragma unroll 2
        for (int t = threadIdx.x; t < kBTile * d / 4; t += blockDim.x) {
            const int j = t / (d / 4), e = (t % (d / 4)) * 4, kj = k0 + j;
            float4 x1 = make_float4(0.f, 0.f, 0.f, 0.f), x2 = x1;
            if (kj < p.L) {
                x1 = *reinterpret_cast<const float4 *>(p.k1 + rix(p, b, kj, h) * d + e);
                x2 = *reinterpret_cast<const float4 *>(p.k2 + ((static_cast<size_t>(b) * p.L + kj) * p.hn + g) * d + e);
            }
            *reinterpret_cast<float4 *>(k1s + j * dk + e) = x1;
            *reinterpret_cast<float4 *>(k2s + j * dk + e) = x2;
        }
#pragma unroll 2
        for (int t = threadIdx.x; t < kBTile * dv / 4; t += blockDim.x) {
            const int j = t / (dv / 4), c = (t % (dv / 4)) * 4, kj = k0 + j;
            *reinterpret_cast<float4 *>(vs + j * dvk + c) =
                kj < p.L ? *reinterpret_cast<const float4 *>(p.v + rix(p, b, kj, h) * dv + c)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
    };
    // scaled logits of key k0 + lane against the warp's rows, both maps
    auto logits = [&](float (&s1)[kRPW], float (&s2)[kRPW]) {
        float a1[kRPW], a2[kRPW];
#pragma unroll
        for (int rr = 0; rr < kRPW; ++rr) a1[rr] = a2[rr] = 0.f;
        const float *k1r = k1s + lane * dk, *k2r = k2s + lane * dk;
#pragma unroll 4
        for (int e4 = 0; e4 < d / 4; ++e4) {
            const float4 x1 = ld4<d>(k1r, e4), x2 = ld4<d>(k2r, e4);
#pragma unroll
            for (int rr = 0; rr < kRPW; ++rr) {
                const int row = warp * kRPW + rr;
                a1[rr] = dot4(ld4<d>(q1s + row * d, e4), x1, a1[rr]);
                a2[rr] = dot4(ld4<d>(q2s + row * d, e4), x2, a2[rr]);
            }
        }
#pragma unroll
        for (int rr = 0; rr < kRPW; ++rr) {
            s1[rr] = a1[rr] * p.scale;
            s2[rr] = a2[rr] * p.scale;
        }
    };
    auto visible = [&](int rr, int k0) {
        const int qi = q0 + warp * kRPW + rr, kj = k0 + lane;
        return qi < p.L && kj < p.L && (!p.causal || kj <= qi);
    };

    // ---- sweep 1: the forward's online softmax (row statistics, O1, O2)
    float m1[kRPW], l1[kRPW], m2[kRPW], l2[kRPW], o1[kRPW][NV], o2[kRPW][NV];
#pragma unroll
    for (int rr = 0; rr < kRPW; ++rr) {
        m1[rr] = m2[rr] = -INFINITY;
        l1[rr] = l2[rr] = 0.f;
#pragma unroll
        for (int c = 0; c < NV; ++c) o1[rr][c] = o2[rr][c] = 0.f;
    }
    const int kv_end = p.causal ? min(p.L, q0 + kBRows) : p.L;
    for (int k0 = 0; k0 < kv_end; k0 += kBTile) {
        load_keys(k0);
        float s1[kRPW], s2[kRPW], w1[kRPW], w2[kRPW];
        logits(s1, s2);
#pragma unroll
        for (int rr = 0; rr < kRPW; ++rr) {
            if (!visible(rr, k0)) s1[rr] = s2[rr] = -INFINITY;
            float al1 = 1.f, al2 = 1.f;
            w1[rr] = w2[rr] = 0.f;
            {
                const float mn = fmaxf(m1[rr], warp_max_b(s1[rr]));
                if (mn != -INFINITY) {
                    al1 = m1[rr] == -INFINITY ? 0.f : expf(m1[rr] - mn);
                    w1[rr] = s1[rr] == -INFINITY ? 0.f : expf(s1[rr] - mn);
                    l1[rr] = l1[rr] * al1 + warp_sum_b(w1[rr]);
                    m1[rr] = mn;
                }
            }
            {
                const float mn = fmaxf(m2[rr], warp_max_b(s2[rr]));
                if (mn != -INFINITY) {
                    al2 = m2[rr] == -INFINITY ? 0.f : expf(m2[rr] - mn);
                    w2[rr] = s2[rr] == -INFINITY ? 0.f : expf(s2[rr] - mn);
                    l2[rr] = l2[rr] * al2 + warp_sum_b(w2[rr]);
                    m2[rr] = mn;
                }
            }
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                o1[rr][c] *= al1;
                o2[rr][c] *= al2;
            }
        }
#pragma unroll 4
        for (int j = 0; j < kBTile; ++j) {
            float pj1[kRPW], pj2[kRPW];
#pragma unroll
            for (int rr = 0; rr < kRPW; ++rr) {
                pj1[rr] = __shfl_sync(0xffffffffu, w1[rr], j);
                pj2[rr] = __shfl_sync(0xffffffffu, w2[rr], j);
            }
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const float vv = vs[j * dvk + lane + 32 * c];
#pragma unroll
                for (int rr = 0; rr < kRPW; ++rr) {
                    o1[rr][c] = fmaf(pj1[rr], vv, o1[rr][c]);
                    o2[rr][c] = fmaf(pj2[rr], vv, o2[rr][c]);
                }
            }
        }
    }

    // ---- do, D1, D2 and the row's dlambda term
    float D1[kRPW], D2[kRPW];
#pragma unroll
    for (int rr = 0; rr < kRPW; ++rr) {
        const int row = warp * kRPW + rr, qi = q0 + row;
        const bool in = qi < p.L;
        float O1[NV], O2[NV], o[NV], dyv[NV];
        float ss = 0.f, dyo = 0.f;
#pragma unroll
        for (int c = 0; c < NV; ++c) {
            O1[c] = in ? o1[rr][c] / l1[rr] : 0.f;
            O2[c] = in ? o2[rr][c] / l2[rr] : 0.f;
            o[c] = O1[c] - lam * O2[c];
            dyv[c] = in ? p.dy[rix(p, b, qi, h) * dv + lane + 32 * c] : 0.f;
            ss = fmaf(o[c], o[c], ss);
            dyo = fmaf(dyv[c], o[c], dyo);
        }
        ss = warp_sum_b(ss);
        dyo = warp_sum_b(dyo);
        float a = in ? 1.f : 0.f, bcoef = 0.f;   // do = a dy - bcoef o (0 on rows past L)
        if (in && !p.no_norm) {
            const float r2 = ss / static_cast<float>(dv) + p.eps;
            const float rms = sqrtf(r2);
            a = (1.f - p.lambda_init) / rms;
            bcoef = a * dyo / (static_cast<float>(dv) * r2);
        }
        float d1 = 0.f, d2 = 0.f;
#pragma unroll
        for (int c = 0; c < NV; ++c) {
            const float dov = a * dyv[c] - bcoef * o[c];
            dos[row * dv + lane + 32 * c] = dov;
            d1 = fmaf(dov, O1[c], d1);
            d2 = fmaf(dov, O2[c], d2);
            if (in) p.dO[rix(p, b, qi, h) * dv + lane + 32 * c] = dov;
        }
        D1[rr] = warp_sum_b(d1);
        D2[rr] = warp_sum_b(d2);
        if (in && lane == 0) {
            float *st = p.stats + rix(p, b, qi, h) * 6;
            st[0] = m1[rr];
            st[1] = l1[rr];
            st[2] = m2[rr];
            st[3] = l2[rr];
            st[4] = D1[rr];
            st[5] = D2[rr];
            p.dlam_row[rix(p, b, qi, h)] = -D2[rr];
        }
    }
    __syncwarp();

    // ---- sweep 2: dq1 and this head's share of dq2
    float dq1a[kRPW][ND], dq2a[kRPW][ND];
#pragma unroll
    for (int rr = 0; rr < kRPW; ++rr)
#pragma unroll
        for (int e = 0; e < ND; ++e) dq1a[rr][e] = dq2a[rr][e] = 0.f;
    for (int k0 = 0; k0 < kv_end; k0 += kBTile) {
        load_keys(k0);
        float s1[kRPW], s2[kRPW], dA[kRPW], ds1[kRPW], ds2[kRPW];
        logits(s1, s2);
#pragma unroll
        for (int rr = 0; rr < kRPW; ++rr) dA[rr] = 0.f;
        const float *vj = vs + lane * dvk;
#pragma unroll 4
        for (int c4 = 0; c4 < dv / 4; ++c4) {
            const float4 x = ld4<dv>(vj, c4);
#pragma unroll
            for (int rr = 0; rr < kRPW; ++rr) dA[rr] = dot4(ld4<dv>(dos + (warp * kRPW + rr) * dv, c4), x, dA[rr]);
        }
#pragma unroll
        for (int rr = 0; rr < kRPW; ++rr) {
            ds1[rr] = ds2[rr] = 0.f;
            if (visible(rr, k0)) {
                const float a1 = expf(s1[rr] - m1[rr]) / l1[rr];
                const float a2 = expf(s2[rr] - m2[rr]) / l2[rr];
                ds1[rr] = a1 * (dA[rr] - D1[rr]);
                ds2[rr] = -lam * a2 * (dA[rr] - D2[rr]);
            }
        }
#pragma unroll 4
        for (int j = 0; j < kBTile; ++j) {
            float x1[kRPW], x2[kRPW];
#pragma unroll
            for (int rr = 0; rr < kRPW; ++rr) {
                x1[rr] = __shfl_sync(0xffffffffu, ds1[rr], j);
                x2[rr] = __shfl_sync(0xffffffffu, ds2[rr], j);
            }
#pragma unroll
            for (int e = 0; e < ND; ++e) {
                const float kk1 = k1s[j * dk + lane + 32 * e], kk2 = k2s[j * dk + lane + 32 * e];
#pragma unroll
                for (int rr = 0; rr < kRPW; ++rr) {
                    dq1a[rr][e] = fmaf(x1[rr], kk1, dq1a[rr][e]);
                    dq2a[rr][e] = fmaf(x2[rr], kk2, dq2a[rr][e]);
                }
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kRPW; ++rr) {
        const int qi = q0 + warp * kRPW + rr;
        if (qi >= p.L) continue;
#pragma unroll
        for (int e = 0; e < ND; ++e) {
            p.dq1[rix(p, b, qi, h) * d + lane + 32 * e] = dq1a[rr][e] * p.scale;
            p.dq2h[rix(p, b, qi, h) * d + lane + 32 * e] = dq2a[rr][e] * p.scale;
        }
    }
}

// ----------------------------------------------------------- column pass --
template <int ND, int NV>
__global__ void __launch_bounds__(kBThreads)
gda_bwd_col_kernel(const BwdParams p) {
    extern __shared__ float sm[];
    constexpr int d = 32 * ND, dv = 32 * NV, dk = d + 4, dvk = dv + 4;
    float *k1s = sm;                       // [kBRows][d]   this CTA's keys (broadcast rows)
    float *k2s = k1s + kBRows * d;         // [kBRows][d]
    float *vks = k2s + kBRows * d;         // [kBRows][dv]
    float *q1s = vks + kBRows * dv;        // [kBTile][d+4]  a tile of query rows (one per lane)
    float *q2s = q1s + kBTile * dk;        // [kBTile][d+4]
    float *dos = q2s + kBTile * dk;        // [kBTile][dv+4]
    float *sts = dos + kBTile * dvk;       // [kBTile][6]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int j0 = blockIdx.x * kBRows;
    const int h = blockIdx.y, b = blockIdx.z;
    const int g = h / (p.hs / p.hn);
    const float lam = p.lambda[h];

    for (int t = threadIdx.x; t < kBRows * d / 4; t += blockDim.x) {
        const int r = t / (d / 4), e = (t % (d / 4)) * 4, kj = j0 + r;
        float4 x1 = make_float4(0.f, 0.f, 0.f, 0.f), x2 = x1;
        if (kj < p.L) {
            x1 = *reinterpret_cast<const float4 *>(p.k1 + rix(p, b, kj, h) * d + e);
            x2 = *reinterpret_cast<const float4 *>(p.k2 + ((static_cast<size_t>(b) * p.L + kj) * p.hn + g) * d + e);
        }
        *reinterpret_cast<float4 *>(k1s + r * d + e) = x1;
        *reinterpret_cast<float4 *>(k2s + r * d + e) = x2;
    }
    for (int t = threadIdx.x; t < kBRows * dv / 4; t += blockDim.x) {
        const int r = t / (dv / 4), c = (t % (dv / 4)) * 4, kj = j0 + r;
        *reinterpret_cast<float4 *>(vks + r * dv + c) =
            kj < p.L ? *reinterpret_cast<const float4 *>(p.v + rix(p, b, kj, h) * dv + c)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    float dva[kRPW][NV], dk1a[kRPW][ND], dk2a[kRPW][ND];
#pragma unroll
    for (int kk = 0; kk < kRPW; ++kk) {
#pragma unroll
        for (int c = 0; c < NV; ++c) dva[kk][c] = 0.f;
#pragma unroll
        for (int e = 0; e < ND; ++e) dk1a[kk][e] = dk2a[kk][e] = 0.f;
    }

    const int i_begin = p.causal ? (j0 / kBTile) * kBTile : 0;
    for (int i0 = i_begin; i0 < p.L; i0 += kBTile) {
        __syncthreads();
#pragma unroll 2
        for (int t = threadIdx.x; t < kBTile * d / 4; t += blockDim.x) {
            const int i = t / (d / 4), e = (t % (d / 4)) * 4, qi = i0 + i;
            float4 x1 = make_float4(0.f, 0.f, 0.f, 0.f), x2 = x1;
            if (qi < p.L) {
                x1 = *reinterpret_cast<const float4 *>(p.q1 + rix(p, b, qi, h) * d + e);
                x2 = *reinterpret_cast<const float4 *>(p.q2 + ((static_cast<size_t>(b) * p.L + qi) * p.hn + g) * d + e);
            }
            *reinterpret_cast<float4 *>(q1s + i * dk + e) = x1;
            *reinterpret_cast<float4 *>(q2s + i * dk + e) = x2;
        }
#pragma unroll 2
        for (int t = threadIdx.x; t < kBTile * dv / 4; t += blockDim.x) {
            const int i = t / (dv / 4), c = (t % (dv / 4)) * 4, qi = i0 + i;
            *reinterpret_cast<float4 *>(dos + i * dvk + c) =
                qi < p.L ? *reinterpret_cast<const float4 *>(p.dO + rix(p, b, qi, h) * dv + c)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int t = threadIdx.x; t < kBTile * 6; t += blockDim.x) {
            const int i = t / 6, qi = i0 + i;
            sts[t] = qi < p.L ? p.stats[rix(p, b, qi, h) * 6 + t % 6] : (t % 6 == 1 || t % 6 == 3 ? 1.f : 0.f);
        }
        __syncthreads();

        // query row i0 + lane against the warp's keys, both maps, and dA
        float a1[kRPW], a2[kRPW], dA[kRPW];
#pragma unroll
        for (int kk = 0; kk < kRPW; ++kk) a1[kk] = a2[kk] = dA[kk] = 0.f;
        {
            const float *q1r = q1s + lane * dk, *q2r = q2s + lane * dk;
#pragma unroll 4
            for (int e4 = 0; e4 < d / 4; ++e4) {
                const float4 y1 = ld4<d>(q1r, e4), y2 = ld4<d>(q2r, e4);
#pragma unroll
                for (int kk = 0; kk < kRPW; ++kk) {
                    const int key = warp * kRPW + kk;
                    a1[kk] = dot4(y1, ld4<d>(k1s + key * d, e4), a1[kk]);
                    a2[kk] = dot4(y2, ld4<d>(k2s + key * d, e4), a2[kk]);
                }
            }
            const float *dor = dos + lane * dvk;
#pragma unroll 4
            for (int c4 = 0; c4 < dv / 4; ++c4) {
                const float4 y = ld4<dv>(dor, c4);
#pragma unroll
                for (int kk = 0; kk < kRPW; ++kk) dA[kk] = dot4(y, ld4<dv>(vks + (warp * kRPW + kk) * dv, c4), dA[kk]);
            }
        }
        const int qi = i0 + lane;
        const float *st = sts + lane * 6;
        float w[kRPW], ds1[kRPW], ds2[kRPW];
#pragma unroll
        for (int kk = 0; kk < kRPW; ++kk) {
            const int kj = j0 + warp * kRPW + kk;
            const bool vis = qi < p.L && kj < p.L && (!p.causal || kj <= qi);
            w[kk] = ds1[kk] = ds2[kk] = 0.f;
            if (vis) {
                const float p1 = expf(a1[kk] * p.scale - st[0]) / st[1];
                const float p2 = expf(a2[kk] * p.scale - st[2]) / st[3];
                w[kk] = p1 - lam * p2;
                ds1[kk] = p1 * (dA[kk] - st[4]);
                ds2[kk] = -lam * p2 * (dA[kk] - st[5]);
            }
        }
#pragma unroll 4
        for (int i = 0; i < kBTile; ++i) {
            float wi[kRPW], x1[kRPW], x2[kRPW];
#pragma unroll
            for (int kk = 0; kk < kRPW; ++kk) {
                wi[kk] = __shfl_sync(0xffffffffu, w[kk], i);
                x1[kk] = __shfl_sync(0xffffffffu, ds1[kk], i);
                x2[kk] = __shfl_sync(0xffffffffu, ds2[kk], i);
            }
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                const float dd = dos[i * dvk + lane + 32 * c];
#pragma unroll
                for (int kk = 0; kk < kRPW; ++kk) dva[kk][c] = fmaf(wi[kk], dd, dva[kk][c]);
            }
#pragma unroll
            for (int e = 0; e < ND; ++e) {
                const float qq1 = q1s[i * dk + lane + 32 * e], qq2 = q2s[i * dk + lane + 32 * e];
#pragma unroll
                for (int kk = 0; kk < kRPW; ++kk) {
                    dk1a[kk][e] = fmaf(x1[kk], qq1, dk1a[kk][e]);
                    dk2a[kk][e] = fmaf(x2[kk], qq2, dk2a[kk][e]);
                }
            }
        }
    }
#pragma unroll
    for (int kk = 0; kk < kRPW; ++kk) {
        const int kj = j0 + warp * kRPW + kk;
        if (kj >= p.L) continue;
#pragma unroll
        for (int c = 0; c < NV; ++c) p.dvo[rix(p, b, kj, h) * dv + lane + 32 * c] = dva[kk][c];
#pragma unroll
        for (int e = 0; e < ND; ++e) {
            p.dk1[rix(p, b, kj, h) * d + lane + 32 * e] = dk1a[kk][e] * p.scale;
            p.dk2h[rix(p, b, kj, h) * d + lane + 32 * e] = dk2a[kk][e] * p.scale;
        }
    }
}

// ---------------------------------------------------------------- reduce --
// Blocks [0, B*L*hn*d / 256): dq2 and dk2 by summing the group's shares;
// the last hs blocks: dlambda_h = sum over (b, i) of the row terms.
__global__ void __launch_bounds__(256)
gda_bwd_reduce_kernel(const BwdParams p, int n_sum_blocks) {
    const int r = p.hs / p.hn;
    if (static_cast<int>(blockIdx.x) < n_sum_blocks) {
        const size_t total = static_cast<size_t>(p.B) * p.L * p.hn * p.d;
        const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        if (t >= total) return;
        const int e = static_cast<int>(t % p.d);
        const size_t bi_g = t / p.d;                  // ((b * L + i) * hn + g)
        const int g = static_cast<int>(bi_g % p.hn);
        const size_t bi = bi_g / p.hn;
        float sq = 0.f, sk = 0.f;
        for (int k = 0; k < r; ++k) {
            const size_t src = (bi * p.hs + g * r + k) * p.d + e;
            sq += p.dq2h[src];
            sk += p.dk2h[src];
        }
        p.dq2[t] = sq;
        p.dk2[t] = sk;
        return;
    }
    __shared__ float red[256];
    const int h = blockIdx.x - n_sum_blocks;
    const size_t rows = static_cast<size_t>(p.B) * p.L;
    float acc = 0.f;
    for (size_t t = threadIdx.x; t < rows; t += blockDim.x) acc += p.dlam_row[t * p.hs + h];
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
        if (static_cast<int>(threadIdx.x) < s) red[threadIdx.x] += red[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) p.dlambda[h] = red[0];
}

template <int ND, int NV>
int launch_bwd(const BwdParams &p, cudaStream_t stream) {
    constexpr int d = 32 * ND, dv = 32 * NV;
    const size_t smem_row = sizeof(float) * (2 * kBRows * d + 2 * kBTile * (d + 4) + kBTile * (dv + 4) + kBRows * dv);
    const size_t smem_col =
        sizeof(float) * (2 * kBRows * d + kBRows * dv + 2 * kBTile * (d + 4) + kBTile * (dv + 4) + kBTile * 6);
    auto rk = gda_bwd_row_kernel<ND, NV>;
    auto ck = gda_bwd_col_kernel<ND, NV>;
    cudaError_t e = cudaFuncSetAttribute(rk, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_row));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_col));
    if (e != cudaSuccess) return record_cuda_error(e);
    const dim3 grid((p.L + kBRows - 1) / kBRows, p.hs, p.B);
    rk<<<grid, kBThreads, smem_row, stream>>>(p);
    ck<<<grid, kBThreads, smem_col, stream>>>(p);
    const size_t total = static_cast<size_t>(p.B) * p.L * p.hn * p.d;
    const int n_sum = static_cast<int>((total + 255) / 256);
    gda_bwd_reduce_kernel<<<n_sum + p.hs, 256, 0, stream>>>(p, n_sum);
    e = cudaGetLastError();
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

}  // namespace

size_t backward_f32_workspace_bytes(int B, int L, int hs, int d, int dv) {
    const size_t rows = static_cast<size_t>(B) * L * hs;
    // stats (6 per row, padded to a multiple of 4) | dO | dq2 shares | dk2 shares | dlambda terms
    return sizeof(float) * ((rows * 6 + 3) / 4 * 4 + rows * (static_cast<size_t>(dv) + 2 * static_cast<size_t>(d) + 1)) +
           256;
}

int launch_backward_f32(const BackwardArgs &a, cudaStream_t stream) {
    BwdParams p;
    p.q1 = a.q1;
    p.k1 = a.k1;
    p.q2 = a.q2;
    p.k2 = a.k2;
    p.v = a.v;
    p.lambda = a.lambda;
    p.dy = a.dy;
    p.dq1 = a.dq1;
    p.dk1 = a.dk1;
    p.dq2 = a.dq2;
    p.dk2 = a.dk2;
    p.dvo = a.dv_out;
    p.dlambda = a.dlambda;
    const size_t rows = static_cast<size_t>(a.B) * a.L * a.hs;
    float *w = static_cast<float *>(a.workspace);
    p.stats = w;
    p.dO = p.stats + (rows * 6 + 3) / 4 * 4;     // 16-byte aligned: read as float4
    p.dq2h = p.dO + rows * a.dv;
    p.dk2h = p.dq2h + rows * a.d;
    p.dlam_row = p.dk2h + rows * a.d;
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
    if (a.hs > 65535 || a.B > 65535) return GDA_ERR_UNSUPPORTED;
    switch (a.d * 1000 + a.dv) {
        case 64 * 1000 + 64: return launch_bwd<2, 2>(p, stream);
        case 64 * 1000 + 128: return launch_bwd<2, 4>(p, stream);
        case 64 * 1000 + 256: return launch_bwd<2, 8>(p, stream);
        case 128 * 1000 + 64: return launch_bwd<4, 2>(p, stream);
        case 128 * 1000 + 128: return launch_bwd<4, 4>(p, stream);
        case 128 * 1000 + 256: return launch_bwd<4, 8>(p, stream);
        default: return GDA_ERR_UNSUPPORTED;
    }
}

}  // namespace gda
