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

constexpr int kBRows = 16;       // query rows (row pass) or keys (column pass) per CTA
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

// -------------------------------------------------------------- row pass --
template <int ND, int NV>   // d = 32 ND, dv = 32 NV
__global__ void __launch_bounds__(kBThreads)
gda_bwd_row_kernel(const BwdParams p) {
    extern __shared__ float sm[];
    constexpr int d = 32 * ND, dv = 32 * NV, dp = d + 1, dvp = dv + 1;
    float *q1s = sm;                       // [kBRows][d]
    float *q2s = q1s + kBRows * d;         // [kBRows][d]
    float *k1s = q2s + kBRows * d;         // [kBTile][d+1]   (+1: a lane per key row, no bank conflicts)
    float *k2s = k1s + kBTile * dp;        // [kBTile][d+1]
    float *vs = k2s + kBTile * dp;         // [kBTile][dv+1]
    float *dos = vs + kBTile * dvp;        // [kBRows][dv]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int q0 = blockIdx.x * kBRows;
    const int h = blockIdx.y, b = blockIdx.z;
    const int g = h / (p.hs / p.hn);
    const float lam = p.lambda[h];

    for (int t = threadIdx.x; t < kBRows * d; t += blockDim.x) {
        const int r = t / d, e = t % d, qi = q0 + r;
        const bool in = qi < p.L;
        q1s[t] = in ? p.q1[rix(p, b, qi, h) * d + e] : 0.f;
        q2s[t] = in ? p.q2[((static_cast<size_t>(b) * p.L + qi) * p.hn + g) * d + e] : 0.f;
    }

    auto load_keys = [&](int k0) {
        __syncthreads();
        for (int t = threadIdx.x; t < kBTile * d; t += blockDim.x) {
            const int j = t / d, e = t % d, kj = k0 + j;
            const bool in = kj < p.L;
            k1s[j * dp + e] = in ? p.k1[rix(p, b, kj, h) * d + e] : 0.f;
            k2s[j * dp + e] = in ? p.k2[((static_cast<size_t>(b) * p.L + kj) * p.hn + g) * d + e] : 0.f;
        }
        for (int t = threadIdx.x; t < kBTile * dv; t += blockDim.x) {
            const int j = t / dv, c = t % dv, kj = k0 + j;
            vs[j * dvp + c] = kj < p.L ? p.v[rix(p, b, kj, h) * dv + c] : 0.f;
        }
        __syncthreads();
    };
    auto logits = [&](int row, int k0, float &s1, float &s2) -> bool {
        const int qi = q0 + row, kj = k0 + lane;
        const bool visible = qi < p.L && kj < p.L && (!p.causal || kj <= qi);
        float a1 = 0.f, a2 = 0.f;
        const float *q1r = q1s + row * d, *q2r = q2s + row * d;
        const float *k1r = k1s + lane * dp, *k2r = k2s + lane * dp;
        #pragma unroll 4
        for (int e = 0; e < d; ++e) {
            a1 = fmaf(q1r[e], k1r[e], a1);
            a2 = fmaf(q2r[e], k2r[e], a2);
        }
        s1 = a1 * p.scale;
        s2 = a2 * p.scale;
        return visible;
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
#pragma unroll
        for (int rr = 0; rr < kRPW; ++rr) {
            const int row = warp * kRPW + rr;
            float s1, s2;
            const bool vis = logits(row, k0, s1, s2);
            if (!vis) s1 = s2 = -INFINITY;
            float w1 = 0.f, w2 = 0.f, al1 = 1.f, al2 = 1.f;
            {
                const float mn = fmaxf(m1[rr], warp_max_b(s1));
                if (mn != -INFINITY) {
                    al1 = m1[rr] == -INFINITY ? 0.f : expf(m1[rr] - mn);
                    w1 = s1 == -INFINITY ? 0.f : expf(s1 - mn);
                    l1[rr] = l1[rr] * al1 + warp_sum_b(w1);
                    m1[rr] = mn;
                }
            }
            {
                const float mn = fmaxf(m2[rr], warp_max_b(s2));
                if (mn != -INFINITY) {
                    al2 = m2[rr] == -INFINITY ? 0.f : expf(m2[rr] - mn);
                    w2 = s2 == -INFINITY ? 0.f : expf(s2 - mn);
                    l2[rr] = l2[rr] * al2 + warp_sum_b(w2);
                    m2[rr] = mn;
                }
            }
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                o1[rr][c] *= al1;
                o2[rr][c] *= al2;
            }
            #pragma unroll 4
            for (int j = 0; j < kBTile; ++j) {
                const float pj1 = __shfl_sync(0xffffffffu, w1, j);
                const float pj2 = __shfl_sync(0xffffffffu, w2, j);
#pragma unroll
                for (int c = 0; c < NV; ++c) {
                    const float vv = vs[j * dvp + lane + 32 * c];
                    o1[rr][c] = fmaf(pj1, vv, o1[rr][c]);
                    o2[rr][c] = fmaf(pj2, vv, o2[rr][c]);
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
#pragma unroll
        for (int rr = 0; rr < kRPW; ++rr) {
            const int row = warp * kRPW + rr;
            float s1, s2;
            const bool vis = logits(row, k0, s1, s2);
            float ds1 = 0.f, ds2 = 0.f;
            if (vis) {
                const float a1 = expf(s1 - m1[rr]) / l1[rr];
                const float a2 = expf(s2 - m2[rr]) / l2[rr];
                float dA = 0.f;
                const float *dor = dos + row * dv, *vj = vs + lane * dvp;
                #pragma unroll 4
                for (int c = 0; c < dv; ++c) dA = fmaf(dor[c], vj[c], dA);
                ds1 = a1 * (dA - D1[rr]);
                ds2 = -lam * a2 * (dA - D2[rr]);
            }
            #pragma unroll 4
            for (int j = 0; j < kBTile; ++j) {
                const float x1 = __shfl_sync(0xffffffffu, ds1, j);
                const float x2 = __shfl_sync(0xffffffffu, ds2, j);
#pragma unroll
                for (int e = 0; e < ND; ++e) {
                    dq1a[rr][e] = fmaf(x1, k1s[j * dp + lane + 32 * e], dq1a[rr][e]);
                    dq2a[rr][e] = fmaf(x2, k2s[j * dp + lane + 32 * e], dq2a[rr][e]);
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
    constexpr int d = 32 * ND, dv = 32 * NV, dp = d + 1, dvp = dv + 1;
    float *k1s = sm;                       // [kBRows][d]   this CTA's keys
    float *k2s = k1s + kBRows * d;         // [kBRows][d]
    float *vks = k2s + kBRows * d;         // [kBRows][dv]
    float *q1s = vks + kBRows * dv;        // [kBTile][d+1] a tile of query rows
    float *q2s = q1s + kBTile * dp;        // [kBTile][d+1]
    float *dos = q2s + kBTile * dp;        // [kBTile][dv+1]
    float *sts = dos + kBTile * dvp;       // [kBTile][6]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int j0 = blockIdx.x * kBRows;
    const int h = blockIdx.y, b = blockIdx.z;
    const int g = h / (p.hs / p.hn);
    const float lam = p.lambda[h];

    for (int t = threadIdx.x; t < kBRows * d; t += blockDim.x) {
        const int r = t / d, e = t % d, kj = j0 + r;
        const bool in = kj < p.L;
        k1s[t] = in ? p.k1[rix(p, b, kj, h) * d + e] : 0.f;
        k2s[t] = in ? p.k2[((static_cast<size_t>(b) * p.L + kj) * p.hn + g) * d + e] : 0.f;
    }
    for (int t = threadIdx.x; t < kBRows * dv; t += blockDim.x) {
        const int r = t / dv, c = t % dv, kj = j0 + r;
        vks[t] = kj < p.L ? p.v[rix(p, b, kj, h) * dv + c] : 0.f;
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
        for (int t = threadIdx.x; t < kBTile * d; t += blockDim.x) {
            const int i = t / d, e = t % d, qi = i0 + i;
            const bool in = qi < p.L;
            q1s[i * dp + e] = in ? p.q1[rix(p, b, qi, h) * d + e] : 0.f;
            q2s[i * dp + e] = in ? p.q2[((static_cast<size_t>(b) * p.L + qi) * p.hn + g) * d + e] : 0.f;
        }
        for (int t = threadIdx.x; t < kBTile * dv; t += blockDim.x) {
            const int i = t / dv, c = t % dv, qi = i0 + i;
            dos[i * dvp + c] = qi < p.L ? p.dO[rix(p, b, qi, h) * dv + c] : 0.f;
        }
        for (int t = threadIdx.x; t < kBTile * 6; t += blockDim.x) {
            const int i = t / 6, qi = i0 + i;
            sts[t] = qi < p.L ? p.stats[rix(p, b, qi, h) * 6 + t % 6] : (t % 6 == 1 || t % 6 == 3 ? 1.f : 0.f);
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kRPW; ++kk) {
            const int key = warp * kRPW + kk, kj = j0 + key;
            const int qi = i0 + lane;
            const bool vis = qi < p.L && kj < p.L && (!p.causal || kj <= qi);
            float w = 0.f, ds1 = 0.f, ds2 = 0.f;
            if (vis) {
                float a1 = 0.f, a2 = 0.f, dA = 0.f;
                const float *q1r = q1s + lane * dp, *q2r = q2s + lane * dp;
                const float *k1r = k1s + key * d, *k2r = k2s + key * d;
                #pragma unroll 4
                for (int e = 0; e < d; ++e) {
                    a1 = fmaf(q1r[e], k1r[e], a1);
                    a2 = fmaf(q2r[e], k2r[e], a2);
                }
                const float *st = sts + lane * 6;
                const float p1 = expf(a1 * p.scale - st[0]) / st[1];
                const float p2 = expf(a2 * p.scale - st[2]) / st[3];
                const float *dor = dos + lane * dvp, *vr = vks + key * dv;
                #pragma unroll 4
                for (int c = 0; c < dv; ++c) dA = fmaf(dor[c], vr[c], dA);
                w = p1 - lam * p2;
                ds1 = p1 * (dA - st[4]);
                ds2 = -lam * p2 * (dA - st[5]);
            }
            #pragma unroll 4
            for (int i = 0; i < kBTile; ++i) {
                const float wi = __shfl_sync(0xffffffffu, w, i);
                const float x1 = __shfl_sync(0xffffffffu, ds1, i);
                const float x2 = __shfl_sync(0xffffffffu, ds2, i);
#pragma unroll
                for (int c = 0; c < NV; ++c) dva[kk][c] = fmaf(wi, dos[i * dvp + lane + 32 * c], dva[kk][c]);
#pragma unroll
                for (int e = 0; e < ND; ++e) {
                    dk1a[kk][e] = fmaf(x1, q1s[i * dp + lane + 32 * e], dk1a[kk][e]);
                    dk2a[kk][e] = fmaf(x2, q2s[i * dp + lane + 32 * e], dk2a[kk][e]);
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
    const size_t smem_row = sizeof(float) * (2 * kBRows * d + 2 * kBTile * (d + 1) + kBTile * (dv + 1) + kBRows * dv);
    const size_t smem_col =
        sizeof(float) * (2 * kBRows * d + kBRows * dv + 2 * kBTile * (d + 1) + kBTile * (dv + 1) + kBTile * 6);
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
    return sizeof(float) * rows * (6 + static_cast<size_t>(dv) + 2 * static_cast<size_t>(d) + 1) + 256;
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
    p.dO = p.stats + rows * 6;
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
