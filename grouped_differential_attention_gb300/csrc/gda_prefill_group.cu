// Grouped prefill for sm_103a: the noise map of each noise head is computed
// ONCE per query tile and key tile and applied to every signal head of its
// group ("Grouped Differential Attention", abstract: few noise-control heads,
// each reused by a group of signal heads akin to grouped-query attention).
//
// Same result as the other prefill kernels:
//   o_h = (softmax(Q1_h K1_h^T / sqrt d) - lambda_h softmax(Q2_g K2_g^T / sqrt d)) V_h
//   y_h = (1 - lambda_init) o_h / sqrt(mean(o_h^2) + eps)
// ("Differential Attention in Large Language Models ...", sections
// "Differential Attention Architecture" and "Headwise Normalization").
//
// Work item = (128-row query tile, batch b, noise head g, S signal heads
// h0 .. h0+S-1 of g's group); S <= 3 divides the group size r.  Each item
// runs two sweeps over its visible keys (64-key tiles), both in one CTA:
//   phase A  every map's row statistics: for the noise map of g and for each
//            of the S signal maps, a running (max, sum) in base-2 units,
//            combined into lse = max + log2(sum).  The noise map is one map
//            of the item, not one per signal head.
//   phase B  per key tile: the noise logits S2 = Q2_g K2_g^T once, their
//            probabilities p2 = 2^(s2 c - lse2) kept in registers; then for
//            each signal head S1_h, P_h = 2^(s1 c - lse1_h) - lambda_h p2 in
//            float32 (one fused multiply-add), rounded once to bf16 and
//            written to shared memory; one P_h V_h product per head into that
//            head's float32 accumulator.  No online rescaling.
// Both maps are normalised before the subtraction (the statistics are exact
// by the end of phase A), so the accumulator holds o_h directly and the
// epilogue only applies the headwise norm.  No statistics leave the SM: no
// workspace.
//
// TMEM (512 columns): accumulators O_h at [128 h, 128 h + 128) for h < S,
// then NSLOT slots of 64 columns for logit tiles (two at S = 3).  A slot is
// released as soon as the compute warps have loaded its tile into registers
// (P goes to shared memory), so the next logit tile's MMA never waits for a
// value product.
// Warp roles (persistent CTA, one per SM):
//   warp 0      TMA producer: Q2 and the S Q1 tiles once per item, a ring of
//               K tiles (one head each) and a ring of V tiles (one head each)
//               in exactly the order the MMAs consume them;
//   warp 1      TMEM allocator and MMA issuer: logit MMAs (SS, K-major) into
//               the slot ring, value MMAs (SS: P from shared memory, V as an
//               MN-major operand) NSLOT uses behind;
//   warps 2-9   compute (thread = query row = TMEM lane; warps 2-5 take key
//               columns 0-31 of each tile, warps 6-9 columns 32-63): running
//               statistics, P, and the epilogue of the item.
// Every mbarrier wait is bounded (1 s) and sets GDA_DEVERR_PREFILL_TIMEOUT.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cmath>

#include "gda.h"
#include "gda_device.cuh"
#include "gda_internal.h"
#include "gda_prefill_common.cuh"

namespace gda {
namespace {

constexpr int kGBN = 64;               // keys per tile
constexpr int kGThreads = 320;         // 10 warps
constexpr int kGComputeWarps = 8;

template <int S> struct GLayout {
    static constexpr int NSLOT = (512 - 128 * S) / 64;   // logit slots of 64 TMEM columns
    static constexpr int LAG = NSLOT;                    // value MMA of use u issued after logit MMA of u + LAG
    static constexpr int KS = 6, VS = 4, NP = 2;         // K, V, P ring depths
    static constexpr int Q_BYTES = kBM * 64 * 2;         // one head's 128 x 64 query tile
    static constexpr int K_BYTES = kGBN * 64 * 2;        // one head's 64 x 64 key tile
    static constexpr int V_BYTES = kGBN * 128 * 2;       // one head's 64 x 128 value tile
    static constexpr int P_BYTES = kBM * kGBN * 2;       // one head's 128 x 64 bf16 P tile
    static constexpr int OFF_Q = 0;                      // Q2, then Q1 of heads h0 .. h0+S-1
    static constexpr int OFF_K = OFF_Q + (S + 1) * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KS * K_BYTES;
    static constexpr int OFF_P = OFF_V + VS * V_BYTES;
    static constexpr int TILES = OFF_P + NP * P_BYTES;
    static_assert(128 * S + 64 * NSLOT <= 512 && NSLOT >= 2, "TMEM budget");
};

struct GCtrl {
    uint64_t q_full, q_empty;
    uint64_t k_full[8], k_empty[8];
    uint64_t v_full[8], v_empty[8];
    uint64_t s_full[6], s_free[6];
    uint64_t p_full[4], p_empty[4];
    uint64_t o_final, o_free, mma_idle;
    uint32_t tmem_base;
    int abort_flag;
    float xm[2][4][kBM];       // [column half][map][row]: phase-A running max
    float xl[2][4][kBM];       // [column half][map][row]: phase-A running sum
    float ss[2][3][kBM];       // [column half][head][row]: epilogue sums of squares
};

template <int S>
constexpr int group_smem_bytes() {
    return GLayout<S>::TILES + static_cast<int>((sizeof(GCtrl) + 1023) / 1024) * 1024 + 1024;
}

struct GParams {
    const float *lambda;
    __nv_bfloat16 *out;
    unsigned *err;
    float lambda_init, eps, scale_log2;
    int B, L, hs, hn, r, nsub, nqt, causal, no_norm;
    int Lk, koff;          // keys per sequence; query row i sits at key position koff + i
};

struct GItem {
    int b, g, h0, q0, nkv;
};

// Items (query tile, b, g, sub-group) with the longest (last) query tiles
// first; round r of the persistent CTAs takes items r*G .. r*G + G-1 in
// snake order, which evens out the causal lengths.
__device__ __forceinline__ bool gitem_of(const GParams &p, int S, int rr, int G, int cid, GItem &it) {
    const int per_tile = p.B * p.hn * p.nsub;
    const long long nitems = static_cast<long long>(p.nqt) * per_tile;
    const int k = (rr & 1) ? (G - 1 - cid) : cid;
    const long long idx = static_cast<long long>(rr) * G + k;
    if (idx >= nitems) return false;
    const int i = static_cast<int>(idx);
    const int qt = p.nqt - 1 - i / per_tile;
    const int rem = i % per_tile;
    it.b = rem / (p.hn * p.nsub);
    const int rem2 = rem % (p.hn * p.nsub);
    it.g = rem2 / p.nsub;
    it.h0 = it.g * p.r + (rem2 % p.nsub) * S;
    it.q0 = qt * kBM;
    const int kv_end = p.causal ? min(p.Lk, p.koff + it.q0 + kBM) : p.Lk;
    it.nkv = (kv_end + kGBN - 1) / kGBN;
    return true;
}

// Per-warp arrival on a barrier that counts the 8 compute warps.
__device__ __forceinline__ void warp_arrive(uint64_t *bar, uint32_t lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

template <int S>
__global__ void __launch_bounds__(kGThreads, 1)
gda_prefill_group_kernel(const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmK1,
                         const __grid_constant__ CUtensorMap tmQ2, const __grid_constant__ CUtensorMap tmK2,
                         const __grid_constant__ CUtensorMap tmV, const GParams p) {
    using LY = GLayout<S>;
    constexpr int NSLOT = LY::NSLOT, LAG = LY::LAG, KS = LY::KS, VS = LY::VS, NP = LY::NP;
    constexpr int M = S + 1;                 // maps per item: noise map (0), signal heads (1..S)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    GCtrl *ctl = reinterpret_cast<GCtrl *>(smem + LY::TILES);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int cid = blockIdx.x;
    const int G = gridDim.x;

    if (threadIdx.x == 0) {
        mbar_init(&ctl->q_full, 1);
        mbar_init(&ctl->q_empty, 1);
        for (int s = 0; s < KS; ++s) {
            mbar_init(&ctl->k_full[s], 1);
            mbar_init(&ctl->k_empty[s], 1);
        }
        for (int s = 0; s < VS; ++s) {
            mbar_init(&ctl->v_full[s], 1);
            mbar_init(&ctl->v_empty[s], 1);
        }
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&ctl->s_full[s], 1);
            mbar_init(&ctl->s_free[s], kGComputeWarps);
        }
        for (int s = 0; s < NP; ++s) {
            mbar_init(&ctl->p_full[s], kGComputeWarps);
            mbar_init(&ctl->p_empty[s], 1);
        }
        mbar_init(&ctl->o_final, 1);
        mbar_init(&ctl->o_free, kGComputeWarps);
        mbar_init(&ctl->mma_idle, 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const uint32_t tSlot0 = 128 * S;          // first logit slot column
    volatile int *abort_flag = &ctl->abort_flag;

    if (warp == 0) {
        // ================================================= TMA producer
        if (elect_one()) {
            tma_prefetch_desc(&tmQ1);
            tma_prefetch_desc(&tmK1);
            tma_prefetch_desc(&tmQ2);
            tma_prefetch_desc(&tmK2);
            tma_prefetch_desc(&tmV);
            uint32_t kt = 0, vt = 0;
            int nq = 0;
            bool ok = true;
            GItem it;
            for (int rr = 0; ok && gitem_of(p, S, rr, G, cid, it); ++rr) {
                if (rr > 0 && !wait_bar(&ctl->q_empty, (rr - 1) & 1, p.err, abort_flag)) break;
                mbar_arrive_expect_tx(&ctl->q_full, M * LY::Q_BYTES);
                tma_load_4d(smem + LY::OFF_Q, &tmQ2, &ctl->q_full, 0, it.g, it.q0, it.b);
#pragma unroll
                for (int h = 0; h < S; ++h)
                    tma_load_4d(smem + LY::OFF_Q + (1 + h) * LY::Q_BYTES, &tmQ1, &ctl->q_full, 0, it.h0 + h, it.q0,
                                it.b);
                ++nq;
                // K tile of map m (0: noise head g, 1..S: signal head h0 + m - 1) at key tile j
                auto load_k = [&](int m, int j) -> bool {
                    const int st = kt % KS;
                    if (kt >= KS && !wait_bar(&ctl->k_empty[st], ((kt / KS) - 1) & 1, p.err, abort_flag))
                        return false;
                    mbar_arrive_expect_tx(&ctl->k_full[st], LY::K_BYTES);
                    if (m == 0)
                        tma_load_4d(smem + LY::OFF_K + st * LY::K_BYTES, &tmK2, &ctl->k_full[st], 0, it.g, j * kGBN,
                                    it.b);
                    else
                        tma_load_4d(smem + LY::OFF_K + st * LY::K_BYTES, &tmK1, &ctl->k_full[st], 0, it.h0 + m - 1,
                                    j * kGBN, it.b);
                    ++kt;
                    return true;
                };
                auto load_v = [&](int h, int j) -> bool {
                    const int st = vt % VS;
                    if (vt >= VS && !wait_bar(&ctl->v_empty[st], ((vt / VS) - 1) & 1, p.err, abort_flag))
                        return false;
                    mbar_arrive_expect_tx(&ctl->v_full[st], LY::V_BYTES);
                    uint8_t *dst = smem + LY::OFF_V + st * LY::V_BYTES;
                    tma_load_4d(dst, &tmV, &ctl->v_full[st], 0, it.h0 + h, j * kGBN, it.b);
                    tma_load_4d(dst + kGBN * 128, &tmV, &ctl->v_full[st], 64, it.h0 + h, j * kGBN, it.b);
                    ++vt;
                    return true;
                };
                // phase A: every map's K tiles, key tile by key tile
                for (int j = 0; ok && j < it.nkv; ++j)
                    for (int m = 0; ok && m < M; ++m) ok = load_k(m, j);
                // phase B: the same K tiles again, with each P-use's V tile LAG uses later
                const int nB = it.nkv * M;
                for (int i = 0; ok && i < nB; ++i) {
                    ok = load_k(i % M, i / M);
                    if (ok && i >= LAG && (i - LAG) % M != 0) ok = load_v((i - LAG) % M - 1, (i - LAG) / M);
                }
                for (int v = (nB > LAG ? nB - LAG : 0); ok && v < nB; ++v)
                    if (v % M != 0) ok = load_v(v % M - 1, v / M);
            }
            // our own copies must land before the CTA may exit
            if (nq > 0) drain_wait(&ctl->q_full, (nq - 1) & 1, p.err);
            for (uint32_t j = (kt > KS ? kt - KS : 0); j < kt; ++j)
                drain_wait(&ctl->k_full[j % KS], (j / KS) & 1, p.err);
            for (uint32_t j = (vt > VS ? vt - VS : 0); j < vt; ++j)
                drain_wait(&ctl->v_full[j % VS], (j / VS) & 1, p.err);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================= MMA issuer
        if (elect_one()) {
            const uint32_t qa0 = smem_u32(smem + LY::OFF_Q);
            const uint32_t ka0 = smem_u32(smem + LY::OFF_K);
            const uint32_t va0 = smem_u32(smem + LY::OFF_V);
            const uint32_t pa0 = smem_u32(smem + LY::OFF_P);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, 128, 1);
            uint32_t u = 0, kt = 0, vt = 0, pk = 0;
            bool ok = true;
            GItem it;
            int nitem = 0;
            // logit MMA of use u, map m, into slot u % NSLOT
            auto qk = [&](int m) -> bool {
                const uint32_t slot = u % NSLOT;
                if (u >= NSLOT && !wait_bar(&ctl->s_free[slot], ((u / NSLOT) - 1) & 1, p.err, abort_flag))
                    return false;
                const uint32_t st = kt % KS;
                if (!wait_bar(&ctl->k_full[st], (kt / KS) & 1, p.err, abort_flag)) return false;
                tc_fence_after();
                issue_qk<64, kGBN>(tmem + tSlot0 + slot * kGBN, qa0 + m * LY::Q_BYTES, ka0 + st * LY::K_BYTES);
                mma_commit(&ctl->s_full[slot]);
                mma_commit(&ctl->k_empty[st]);
                ++u;
                ++kt;
                return true;
            };
            bool first_pv = true;
            // value MMA of P-use v (phase-B index) of the current item: O_h += P_h V_h
            auto pv = [&](int v) -> bool {
                const int h = v % (S + 1) - 1, j = v / (S + 1);
                const uint32_t buf = pk % NP;
                if (!wait_bar(&ctl->p_full[buf], (pk / NP) & 1, p.err, abort_flag)) return false;
                const uint32_t st = vt % VS;
                if (!wait_bar(&ctl->v_full[st], (vt / VS) & 1, p.err, abort_flag)) return false;
                if (first_pv) {
                    // the accumulators are free once the previous item's epilogue has read them
                    if (nitem > 0 && !wait_bar(&ctl->o_free, (nitem - 1) & 1, p.err, abort_flag)) return false;
                    first_pv = false;
                }
                tc_fence_after();
                const uint32_t pa = pa0 + buf * LY::P_BYTES, va = va0 + st * LY::V_BYTES;
#pragma unroll
                for (int k = 0; k < kGBN / 16; ++k) {
                    const uint64_t a = smem_desc_sw128(pa + k * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(va + k * 2048, kGBN * 128, 1024);
                    mma_ss(tmem + 128 * h, a, b, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&ctl->p_empty[buf]);
                mma_commit(&ctl->v_empty[st]);
                ++pk;
                ++vt;
                return true;
            };
            for (int rr = 0; ok && gitem_of(p, S, rr, G, cid, it); ++rr) {
                if (!wait_bar(&ctl->q_full, rr & 1, p.err, abort_flag)) break;
                for (int j = 0; ok && j < it.nkv; ++j)
                    for (int m = 0; ok && m < M; ++m) ok = qk(m);
                const int nB = it.nkv * M;
                first_pv = true;
                for (int i = 0; ok && i < nB; ++i) {
                    ok = qk(i % M);
                    if (ok && i == nB - 1) mma_commit(&ctl->q_empty);     // the item's last logit MMA
                    if (ok && i >= LAG && (i - LAG) % M != 0) ok = pv(i - LAG);
                }
                for (int v = (nB > LAG ? nB - LAG : 0); ok && v < nB; ++v)
                    if (v % M != 0) ok = pv(v);
                if (!ok) break;
                mma_commit(&ctl->o_final);
                ++nitem;
            }
            // every issued MMA completes before TMEM is released
            mma_commit(&ctl->mma_idle);
            drain_wait(&ctl->mma_idle, 0, p.err);
        }
        __syncwarp();
    } else {
        // ================================================= compute warps
        const int half = (warp - 2) / 4;          // key columns [32 half, 32 half + 32) of every tile
        const int quarter = warp % 4;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t pair_bar = 1 + quarter;    // the two warps that hold this row's halves
        const float sl2 = p.scale_log2;
        uint8_t *pbase = smem + LY::OFF_P;
        uint32_t u = 0, pk = 0;
        GItem it;
        for (int rr = 0; gitem_of(p, S, rr, G, cid, it); ++rr) {
            const int qrow = it.q0 + row;
            const bool in = qrow < p.L;
            const int last_key = p.causal ? min(p.koff + qrow, p.Lk - 1) : p.Lk - 1;
            float lam[S];
#pragma unroll
            for (int h = 0; h < S; ++h) lam[h] = p.lambda[it.h0 + h];
            bool ok = true;

            // load this thread's 32 logits of use u into rr; release the slot
            auto load_use = [&](uint32_t (&x)[32]) {
                const uint32_t slot = u % NSLOT;
                if (!warp_wait(&ctl->s_full[slot], (u / NSLOT) & 1, p.err, abort_flag)) ok = false;
                tc_fence_after();
                tmem_ld32(tmem + lane_off + tSlot0 + slot * kGBN + half * 32, x);
                tmem_ld_wait_regs(x);
                tc_fence_before();
                warp_arrive(&ctl->s_free[slot], lane);
                ++u;
            };

            // ---------------------------------------------- phase A: row statistics
            float mx[M], ls[M];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                mx[m] = -INFINITY;
                ls[m] = 0.f;
            }
            for (int j = 0; j < it.nkv; ++j) {
                const int k0 = j * kGBN + half * 32;
                const bool need_mask = k0 + 31 > last_key;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    uint32_t x[32];
                    load_use(x);
                    if (need_mask) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (k0 + e > last_key) x[e] = __float_as_uint(-INFINITY);
                    }
                    float m4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) m4[i] = __uint_as_float(x[i]);
#pragma unroll
                    for (int e = 4; e < 32; e += 8)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            m4[i] = max3f(m4[i], __uint_as_float(x[e + 2 * i]), __uint_as_float(x[e + 2 * i + 1]));
                    const float tmax = max3f(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2;
                    const float mn = fmaxf(mx[m], tmax);
                    if (mn != -INFINITY) {
                        const float neg = -mn;
                        float sa = 0.f, sb = 0.f, sc = 0.f, sd = 0.f;
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            float x0 = __uint_as_float(x[e]), x1 = __uint_as_float(x[e + 1]);
                            float x2 = __uint_as_float(x[e + 2]), x3 = __uint_as_float(x[e + 3]);
                            ffma2(x0, x1, sl2, sl2, neg, neg);
                            ffma2(x2, x3, sl2, sl2, neg, neg);
                            fadd2(sa, sb, fast_exp2(x0), fast_exp2(x1));
                            fadd2(sc, sd, fast_exp2(x2), fast_exp2(x3));
                        }
                        ls[m] = ls[m] * fast_exp2(mx[m] - mn) + ((sa + sb) + (sc + sd));
                        mx[m] = mn;
                    }
                }
            }
            // combine the two column halves of the row: lse = max + log2(sum), base 2
#pragma unroll
            for (int m = 0; m < M; ++m) {
                ctl->xm[half][m][row] = mx[m];
                ctl->xl[half][m][row] = ls[m];
            }
            named_bar_sync(pair_bar, 64);
            float nlse[M];                        // -lse of each map (-inf for rows past L: every P is 0)
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const float m0 = ctl->xm[0][m][row], m1 = ctl->xm[1][m][row];
                const float mm = fmaxf(m0, m1);
                float lsum = 0.f;
                if (m0 != -INFINITY) lsum += ctl->xl[0][m][row] * fast_exp2(m0 - mm);
                if (m1 != -INFINITY) lsum += ctl->xl[1][m][row] * fast_exp2(m1 - mm);
                nlse[m] = in ? -(mm + __log2f(lsum)) : -INFINITY;
            }

            // ---------------------------------------------- phase B: P_h = A1_h - lambda_h A2, P_h V_h
            for (int j = 0; j < it.nkv; ++j) {
                const int k0 = j * kGBN + half * 32;
                const bool need_mask = k0 + 31 > last_key;
                float p2[32];
                {
                    uint32_t x[32];
                    load_use(x);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float y0 = __uint_as_float(x[e]), y1 = __uint_as_float(x[e + 1]);
                        ffma2(y0, y1, sl2, sl2, nlse[0], nlse[0]);
                        p2[e] = fast_exp2(y0);
                        p2[e + 1] = fast_exp2(y1);
                    }
                }
#pragma unroll
                for (int h = 0; h < S; ++h) {
                    uint32_t x[32];
                    load_use(x);
                    const float nl = nlse[1 + h], nlam = -lam[h];
                    uint32_t pw[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float y0 = __uint_as_float(x[e]), y1 = __uint_as_float(x[e + 1]);
                        ffma2(y0, y1, sl2, sl2, nl, nl);
                        float q0 = fmaf(nlam, p2[e], fast_exp2(y0));
                        float q1 = fmaf(nlam, p2[e + 1], fast_exp2(y1));
                        if (need_mask) {
                            if (k0 + e > last_key) q0 = 0.f;
                            if (k0 + e + 1 > last_key) q1 = 0.f;
                        }
                        pw[e / 2] = pack_bf16x2(q0, q1);
                    }
                    // P tile in the K-major 128-byte-swizzled layout of the value MMA's
                    // A operand: 16-byte chunk c of row t at chunk c ^ (t % 8)
                    const uint32_t buf = pk % NP;
                    if (pk >= NP && !warp_wait(&ctl->p_empty[buf], ((pk / NP) - 1) & 1, p.err, abort_flag))
                        ok = false;
                    uint8_t *prow = pbase + buf * LY::P_BYTES + row * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int ch = half * 4 + c;
                        *reinterpret_cast<uint4 *>(prow + ((ch ^ (row & 7)) << 4)) =
                            make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                    }
                    fence_proxy_async_smem();
                    warp_arrive(&ctl->p_full[buf], lane);
                    ++pk;
                }
            }

            // ---------------------------------------------- epilogue: headwise norm of each head
            ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
            if (ok) ok = warp_wait(&ctl->o_final, rr & 1, p.err, abort_flag);
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < S; ++h) {
                float ss = 0.f;
                if (ok) {
                    const uint32_t tO = tmem + lane_off + 128 * h + half * 64;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + cc * 32, o);
                        tmem_ld_wait_regs(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ss = fmaf(__uint_as_float(o[e]), __uint_as_float(o[e]), ss);
                    }
                }
                ctl->ss[half][h][row] = ss;
            }
            named_bar_sync(pair_bar, 64);
            ok = __all_sync(0xffffffffu, ok);
#pragma unroll
            for (int h = 0; h < S; ++h) {
                const float ss_tot = ctl->ss[0][h][row] + ctl->ss[1][h][row];
                const float yscale = p.no_norm ? 1.f : (1.f - p.lambda_init) * rsqrtf(ss_tot / 128.f + p.eps);
                if (ok) {
                    const uint32_t tO = tmem + lane_off + 128 * h + half * 64;
                    __nv_bfloat16 *orow =
                        p.out + ((static_cast<size_t>(it.b) * p.L + qrow) * p.hs + it.h0 + h) * 128 + half * 64;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(tO + cc * 32, o);
                        tmem_ld_wait_regs(o);
                        uint32_t pko[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2)
                            pko[e / 2] = pack_bf16x2(__uint_as_float(o[e]) * yscale, __uint_as_float(o[e + 1]) * yscale);
                        if (in) {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4)
                                dst[v4] = make_uint4(pko[4 * v4], pko[4 * v4 + 1], pko[4 * v4 + 2], pko[4 * v4 + 3]);
                        }
                    }
                }
            }
            // the accumulators may now be overwritten by the next item's first value MMA
            tc_fence_before();
            warp_arrive(&ctl->o_free, lane);
            // both warps of the pair agree on whether to go on (pairs share no named barrier)
            if (bar_red_or(pair_bar, 64, !ok || *abort_flag)) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Signal heads per item: the largest divisor of the group size r that is at most 3.
int heads_per_item(int r) {
    for (int s = 3; s >= 1; --s)
        if (r % s == 0) return s;
    return 1;
}

template <int S>
int launch_group_impl(const PrefillArgs &a, cudaStream_t stream) {
    CUtensorMap mQ1, mK1, mQ2, mK2, mV;
    const uint64_t B = a.B, L = a.L, Lk = a.Lk > 0 ? a.Lk : a.L, hs = a.hs, hn = a.hn;
    {
        const uint64_t dq[4] = {64, hs, L, B}, dk[4] = {64, hs, Lk, B};
        const uint64_t sq[3] = {128, hs * 128, L * hs * 128}, sk[3] = {128, hs * 128, Lk * hs * 128};
        const uint32_t boxq[4] = {64, 1, kBM, 1}, boxk[4] = {64, 1, kGBN, 1};
        if (!encode_tmap_4d_bf16(&mQ1, a.q1, dq, sq, boxq)) return GDA_ERR_CUDA;
        if (!encode_tmap_4d_bf16(&mK1, a.k1, dk, sk, boxk)) return GDA_ERR_CUDA;
    }
    {
        const uint64_t dq[4] = {64, hn, L, B}, dk[4] = {64, hn, Lk, B};
        const uint64_t sq[3] = {128, hn * 128, L * hn * 128}, sk[3] = {128, hn * 128, Lk * hn * 128};
        const uint32_t boxq[4] = {64, 1, kBM, 1}, boxk[4] = {64, 1, kGBN, 1};
        if (!encode_tmap_4d_bf16(&mQ2, a.q2, dq, sq, boxq)) return GDA_ERR_CUDA;
        if (!encode_tmap_4d_bf16(&mK2, a.k2, dk, sk, boxk)) return GDA_ERR_CUDA;
    }
    {
        const uint64_t dv4[4] = {128, hs, Lk, B};
        const uint64_t sv[3] = {256, hs * 256, Lk * hs * 256};
        const uint32_t box[4] = {64, 1, kGBN, 1};
        if (!encode_tmap_4d_bf16(&mV, a.v, dv4, sv, box)) return GDA_ERR_CUDA;
    }
    GParams p;
    p.lambda = a.lambda;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.err = a.dev_err;
    p.lambda_init = a.lambda_init;
    p.eps = a.eps;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / 8.0);   // log2(e) / sqrt(64)
    p.B = a.B;
    p.L = a.L;
    p.hs = a.hs;
    p.hn = a.hn;
    p.r = a.hs / a.hn;
    p.nsub = p.r / S;
    p.nqt = (a.L + kBM - 1) / kBM;
    p.causal = a.causal;
    p.no_norm = (a.flags & GDA_FLAG_NO_NORM) ? 1 : 0;
    p.Lk = static_cast<int>(Lk);
    p.koff = static_cast<int>(Lk) - a.L;

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    auto kern = gda_prefill_group_kernel<S>;
    constexpr int smem = group_smem_bytes<S>();
    static_assert(smem <= 232448, "shared memory budget");
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return record_cuda_error(e);
    const long long nitems = static_cast<long long>(p.nqt) * a.B * a.hn * p.nsub;
    if (nitems <= 0 || nitems > 0x7fffffffLL) return GDA_ERR_UNSUPPORTED;
    long long grid = sms;
    if (grid > nitems) grid = nitems;
    kern<<<static_cast<unsigned>(grid), kGThreads, smem, stream>>>(mQ1, mK1, mQ2, mK2, mV, p);
    e = cudaGetLastError();
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

}  // namespace

bool prefill_group_supported(const PrefillArgs &a) { return a.d == 64 && a.dv == 128; }

int launch_prefill_group(const PrefillArgs &a, cudaStream_t stream) {
    if (!prefill_group_supported(a)) return GDA_ERR_UNSUPPORTED;
    switch (heads_per_item(a.hs / a.hn)) {
        case 3: return launch_group_impl<3>(a, stream);
        case 2: return launch_group_impl<2>(a, stream);
        default: return launch_group_impl<1>(a, stream);
    }
}

}  // namespace gda
