// Two-pass grouped differential attention prefill for sm_103a: the
// difference map is formed before the value product.  Also serves chunked
// prefill (L query rows continuing a sequence of Lk >= L keys: query row i
// sits at key position Lk - L + i).
//
// Same result as the single-pass kernel (gda_prefill_tc.cu):
//   o = softmax(Q1_h K1_h^T / sqrt d) V_h - lambda_h softmax(Q2_g K2_g^T / sqrt d) V_h
//   y = (1 - lambda_init) o / sqrt(mean(o^2) + eps)
// ("Differential Attention in Large Language Models ...", sections
// "Differential Attention Architecture" and "Headwise Normalization"; noise
// heads shared by groups per the "Grouped Differential Attention" abstract),
// computed as o = (A1 - lambda_h A2) V_h with the maps' final statistics known
// up front:
//   pass 1 (gda_lse_tc_kernel): for every query row and every head of either
//     map, lse = log2 sum_j 2^(s_j log2(e) / sqrt d) over the row's visible
//     keys, in base-2 units (the noise map once per noise head, not once per
//     signal head).  Written to a float32 workspace [B, h_s + h_n, L].
//   pass 2 (gda_diffmap_tc_kernel): per (128-row query tile, b, h), both logit
//     tiles on the tensor core, P = 2^(s1 c - lse1) - lambda_h 2^(s2 c - lse2)
//     (c = log2(e) / sqrt d) rounded once to bf16, and ONE PV product into one
//     float32 accumulator.  No online rescaling; the epilogue only applies the
//     headwise norm.
// One accumulator of dv columns per CTA: dv = 256 fits one CTA's TMEM next to
// the double-buffered S tiles (256 + 4 x 64 = 512 columns).
//
// Both kernels are persistent with the single-pass kernel's roles: warp 0 TMA
// producer, warp 1 TMEM allocator and MMA issuer, warps 2-9 the softmax
// threads (thread = query row = TMEM lane; warps 2-5 take key columns 0-31 of
// each 64-key tile, warps 6-9 columns 32-63).  Every wait is bounded (1 s)
// and sets GDA_DEVERR_PREFILL_TIMEOUT on expiry.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cmath>
#include <type_traits>

#include "gda.h"
#include "gda_device.cuh"
#include "gda_internal.h"
#include "gda_prefill_common.cuh"

namespace gda {
namespace {

// Bounded wait that first polls without the suspend-time hint (a wait whose phase has
// already completed costs about a third as much that way, which matters on the
// single-thread MMA issuer), then falls back to the bounded hinted wait.
__device__ __forceinline__ bool wait_quick(uint64_t *bar, uint32_t parity, unsigned *err, volatile int *abort) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0 || wait_bar(bar, parity, err, abort);
}

constexpr int kWarps2 = 10;
constexpr int kThreads2 = 32 * kWarps2;
constexpr int kSmThreads = 256;     // softmax threads (8 warps)
constexpr int kBN2 = 64;            // keys per tile

struct P2Params {
    const float *lambda;
    float *lse;                     // [B, hs + hn, lse_ld] (base-2 log-sum-exp)
    __nv_bfloat16 *out;
    unsigned *err;
    float lambda_init, eps, scale_log2;
    int B, L, hs, hn, dv, causal, nqt, no_norm;
    int lse_ld;                     // row stride of lse (>= L)
    int Lk, koff;                   // keys per sequence; query row i sits at key position koff + i
};

// ---------------------------------------------------------------- items --
// Pass 1 item = (query tile, batch, head of either map): head < hs is signal
// head `head`, head >= hs noise head head - hs.  Pass 2 item = (query tile,
// batch, signal head).  Longest (last) query tiles first; snake order over
// the persistent CTAs evens out the causal lengths.
struct Item2 {
    int b, head, q0, nkv;
};

__device__ __forceinline__ bool item2_of(const P2Params &p, int heads, int r, int G, int cid, Item2 &it) {
    const int per_tile = p.B * heads;
    const long long nitems = static_cast<long long>(p.nqt) * per_tile;
    const int k = (r & 1) ? (G - 1 - cid) : cid;
    const long long idx = static_cast<long long>(r) * G + k;
    if (idx >= nitems) return false;
    const int i = static_cast<int>(idx);
    const int qt = p.nqt - 1 - i / per_tile;
    const int rem = i % per_tile;
    it.b = rem / heads;
    it.head = rem % heads;
    it.q0 = qt * kBM;
    const int kv_end = p.causal ? min(p.Lk, p.koff + it.q0 + kBM) : p.Lk;
    it.nkv = (kv_end + kBN2 - 1) / kBN2;
    return true;
}

// =========================================================== pass 1: lse ==

template <int D> struct LseLayout {
    static constexpr int KS = 4;
    static constexpr int Q_BYTES = kBM * D * 2;
    static constexpr int K_BYTES = kBN2 * D * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = Q_BYTES;
    static constexpr int TILES = OFF_K + KS * K_BYTES;
};

struct LseCtrl {
    uint64_t q_full, q_empty;
    uint64_t k_full[4], k_empty[4];
    uint64_t s_full[2], s_free[2];
    uint64_t mma_idle;
    uint32_t tmem_base;
    int abort_flag;
    float part_m[2][2][kBM];      // [item parity][column half][row]
    float part_l[2][2][kBM];
};

template <int D>
constexpr int lse_smem_bytes() {
    return LseLayout<D>::TILES + static_cast<int>((sizeof(LseCtrl) + 1023) / 1024) * 1024 + 1024;
}

template <int D>
__global__ void __launch_bounds__(kThreads2, 2)
gda_lse_tc_kernel(const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmK1,
                  const __grid_constant__ CUtensorMap tmQ2, const __grid_constant__ CUtensorMap tmK2,
                  const P2Params p) {
    using LY = LseLayout<D>;
    constexpr int KS = LY::KS;
    const int heads = p.hs + p.hn;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, offset from the shared array itself so that accesses stay in the
    // shared state space (32-bit addresses)
    uint8_t *smem = smem_raw + ((0u - smem_u32(smem_raw)) & 1023u);
    LseCtrl *ctl = reinterpret_cast<LseCtrl *>(smem + LY::TILES);
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
        for (int bb = 0; bb < 2; ++bb) {
            mbar_init(&ctl->s_full[bb], 1);
            mbar_init(&ctl->s_free[bb], kSmThreads);
        }
        mbar_init(&ctl->mma_idle, 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (elect_one()) {
            tma_prefetch_desc(&tmQ1);
            tma_prefetch_desc(&tmK1);
            tma_prefetch_desc(&tmQ2);
            tma_prefetch_desc(&tmK2);
            uint32_t kt = 0;
            int nq = 0;
            bool ok = true;
            Item2 it;
            for (int r = 0; ok && item2_of(p, heads, r, G, cid, it); ++r) {
                const bool sig = it.head < p.hs;
                const void *tq = sig ? static_cast<const void *>(&tmQ1) : static_cast<const void *>(&tmQ2);
                const void *tk = sig ? static_cast<const void *>(&tmK1) : static_cast<const void *>(&tmK2);
                const int hh = sig ? it.head : it.head - p.hs;
                if (r > 0 && !wait_quick(&ctl->q_empty, (r - 1) & 1, p.err, abort_flag)) break;
                mbar_arrive_expect_tx(&ctl->q_full, LY::Q_BYTES);
#pragma unroll
                for (int blk = 0; blk < D / 64; ++blk)
                    tma_load_4d(smem + LY::OFF_Q + blk * kBM * 128, tq, &ctl->q_full, blk * 64, hh, it.q0, it.b);
                ++nq;
                int kdone = 0;
                for (int j = 0; j < it.nkv; ++j) {
                    const uint32_t gk = kt + j;
                    const int st = gk % KS;
                    if (gk >= KS && !wait_quick(&ctl->k_empty[st], ((gk / KS) - 1) & 1, p.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sb = smem + LY::OFF_K + st * LY::K_BYTES;
                    mbar_arrive_expect_tx(&ctl->k_full[st], LY::K_BYTES);
#pragma unroll
                    for (int blk = 0; blk < D / 64; ++blk)
                        tma_load_4d(sb + blk * kBN2 * 128, tk, &ctl->k_full[st], blk * 64, hh, j * kBN2, it.b);
                    ++kdone;
                }
                kt += kdone;
            }
            if (nq > 0) drain_wait(&ctl->q_full, (nq - 1) & 1, p.err);
            for (uint32_t j = (kt > KS ? kt - KS : 0); j < kt; ++j)
                drain_wait(&ctl->k_full[j % KS], (j / KS) & 1, p.err);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (elect_one()) {
            const uint32_t qa = smem_u32(smem + LY::OFF_Q);
            const uint32_t k0a = smem_u32(smem + LY::OFF_K);
            uint32_t kt = 0, gt = 0;
            bool ok = true;
            Item2 it;
            for (int r = 0; ok && item2_of(p, heads, r, G, cid, it); ++r) {
                if (!wait_quick(&ctl->q_full, r & 1, p.err, abort_flag)) break;
                for (int j = 0; j < it.nkv; ++j) {
                    const uint32_t gk = kt + j, gs = gt + j;
                    const int bb = gs & 1;
                    const uint32_t u = gs >> 1;
                    if (!wait_quick(&ctl->k_full[gk % KS], (gk / KS) & 1, p.err, abort_flag)) { ok = false; break; }
                    if (u >= 1 && !wait_quick(&ctl->s_free[bb], (u - 1) & 1, p.err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    issue_qk<D, kBN2>(tmem + bb * kBN2, qa, k0a + (gk % KS) * LY::K_BYTES);
                    mma_commit(&ctl->s_full[bb]);
                    mma_commit(&ctl->k_empty[gk % KS]);
                }
                if (!ok) break;
                mma_commit(&ctl->q_empty);
                kt += it.nkv;
                gt += it.nkv;
            }
            mma_commit(&ctl->mma_idle);
            drain_wait(&ctl->mma_idle, 0, p.err);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ row statistics
        const int half = (warp - 2) / 4;          // key columns [32 half, 32 half + 32) of a tile
        const int quarter = warp % 4;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        uint32_t gt = 0;
        Item2 it;
        for (int r = 0; item2_of(p, heads, r, G, cid, it); ++r) {
            const int qrow = it.q0 + row;
            const int last_key = p.causal ? min(p.koff + qrow, p.Lk - 1) : p.Lk - 1;
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < it.nkv; ++j) {
                const uint32_t gs = gt + j;
                const int bb = gs & 1;
                // per-lane wait: a failed one sets the error word and the flag that ends every
                // later wait at once; the loop runs on, so the barrier counts stay whole
                if (!wait_quick(&ctl->s_full[bb], (gs >> 1) & 1, p.err, abort_flag)) ok = false;
                tc_fence_after();
                uint32_t rr[32];
                tmem_ld32(tmem + lane_off + bb * kBN2 + half * 32, rr);
                tmem_ld_wait_regs(rr);
                tc_fence_before();
                mbar_arrive(&ctl->s_free[bb]);     // the tile is in registers
                const int k0 = j * kBN2 + half * 32;
                if (k0 + 31 > last_key) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (k0 + e > last_key) rr[e] = __float_as_uint(-INFINITY);
                }
                float mx4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) mx4[i] = __uint_as_float(rr[i]);
#pragma unroll
                for (int e = 4; e < 32; e += 8)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        mx4[i] = max3f(mx4[i], __uint_as_float(rr[e + 2 * i]), __uint_as_float(rr[e + 2 * i + 1]));
                const float mx = max3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3])) * sl2;
                const float mn = fmaxf(m, mx);
                if (mn != -INFINITY) {
                    const float neg = -mn;
                    float sa = 0.f, sb = 0.f, sc = 0.f, sd = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        float x0 = __uint_as_float(rr[e]), x1 = __uint_as_float(rr[e + 1]);
                        float x2 = __uint_as_float(rr[e + 2]), x3 = __uint_as_float(rr[e + 3]);
                        ffma2(x0, x1, sl2, sl2, neg, neg);
                        ffma2(x2, x3, sl2, sl2, neg, neg);
                        fadd2(sa, sb, fast_exp2(x0), fast_exp2(x1));
                        fadd2(sc, sd, fast_exp2(x2), fast_exp2(x3));
                    }
                    l = l * fast_exp2(m - mn) + ((sa + sb) + (sc + sd));
                    m = mn;
                }
            }
            // combine the two column halves; half 0 writes the row's lse
            const int pb = r & 1;
            ctl->part_m[pb][half][row] = m;
            ctl->part_l[pb][half][row] = l;
            named_bar_sync(1, kSmThreads);
            if (half == 0 && qrow < p.L && ok) {
                const float m0 = ctl->part_m[pb][0][row], m1 = ctl->part_m[pb][1][row];
                const float mm = fmaxf(m0, m1);
                const float ls = ctl->part_l[pb][0][row] * fast_exp2(m0 - mm) +
                                 (m1 == -INFINITY ? 0.f : ctl->part_l[pb][1][row] * fast_exp2(m1 - mm));
                p.lse[(static_cast<size_t>(it.b) * heads + it.head) * p.lse_ld + qrow] = mm + __log2f(ls);
            }
            gt += it.nkv;
            if (bar_red_or(1, kSmThreads, !ok || *abort_flag)) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// ====================================================== pass 2: diff map ==

template <int D, int DV> struct DmCfg;
template <> struct DmCfg<64, 128> { static constexpr int KS = 4, VS = 4; };
template <> struct DmCfg<64, 256> { static constexpr int KS = 4, VS = 3; };
template <> struct DmCfg<128, 128> { static constexpr int KS = 3, VS = 3; };
template <> struct DmCfg<128, 256> { static constexpr int KS = 2, VS = 2; };

template <int D, int DV> struct DmLayout {
    static constexpr int KS = DmCfg<D, DV>::KS;
    static constexpr int VS = DmCfg<D, DV>::VS;
    static constexpr int Q_BYTES = kBM * D * 2;
    static constexpr int K_BYTES = kBN2 * D * 2;       // one of K1 / K2
    static constexpr int KST_BYTES = 2 * K_BYTES;      // K stage: K1 then K2
    static constexpr int V_BYTES = kBN2 * DV * 2;      // V stage: DV / 64 column blocks
    static constexpr int OFF_Q1 = 0;
    static constexpr int OFF_Q2 = Q_BYTES;
    static constexpr int OFF_K = 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KS * KST_BYTES;
    static constexpr int TILES = OFF_V + VS * V_BYTES;
    static_assert(DV + 4 * kBN2 <= 512, "TMEM budget");
};

struct DmCtrl {
    uint64_t q_full, q_empty;
    uint64_t k_full[4], k_empty[4];
    uint64_t v_full[4], v_empty[4];
    uint64_t s_full[2];           // both logit tiles of an S buffer are in TMEM
    uint64_t p_full[2];           // P of an S buffer is in TMEM (both column halves)
    uint64_t o_final, o_free, mma_idle;
    uint32_t tmem_base;
    int abort_flag;
    float ss_part[2][kBM];        // [column half][row]
};

template <int D, int DV>
constexpr int dm_smem_bytes() {
    return DmLayout<D, DV>::TILES + static_cast<int>((sizeof(DmCtrl) + 1023) / 1024) * 1024 + 1024;
}

// O += P V for one 64-key tile.  P is bf16 pairs in TMEM: keys 0-31 in
// columns tP .. tP+15 and keys 32-63 in tP+32 .. tP+47 (each column half
// writes over the S columns it alone read).  V stage: DV/64 MN-major column
// blocks of [64 keys x 64] with 128-byte rows, 128-byte swizzle.
template <int DV>
__device__ __forceinline__ void issue_pv_split(uint32_t tO, uint32_t tP, uint32_t va, bool acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, DV, 1);
#pragma unroll
    for (int k = 0; k < kBN2 / 16; ++k) {
        const uint64_t b = smem_desc_sw128(va + k * 2048, kBN2 * 128, 1024);
        mma_ts(tO, tP + (k / 2) * 32 + (k % 2) * 8, b, idesc, (acc || k > 0) ? 1u : 0u);
    }
}

template <int D, int DV>
__global__ void __launch_bounds__(kThreads2, 1)
gda_diffmap_tc_kernel(const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmK1,
                      const __grid_constant__ CUtensorMap tmQ2, const __grid_constant__ CUtensorMap tmK2,
                      const __grid_constant__ CUtensorMap tmV, const P2Params p) {
    using LY = DmLayout<D, DV>;
    constexpr int KS = LY::KS;
    constexpr int VS = LY::VS;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, offset from the shared array itself so that accesses stay in the
    // shared state space (32-bit addresses)
    uint8_t *smem = smem_raw + ((0u - smem_u32(smem_raw)) & 1023u);
    DmCtrl *ctl = reinterpret_cast<DmCtrl *>(smem + LY::TILES);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int cid = blockIdx.x;
    const int G = gridDim.x;
    const int r_grp = p.hs / p.hn;

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
        for (int bb = 0; bb < 2; ++bb) {
            mbar_init(&ctl->s_full[bb], 1);
            mbar_init(&ctl->p_full[bb], kSmThreads);
        }
        mbar_init(&ctl->o_final, 1);
        mbar_init(&ctl->o_free, kSmThreads);
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
    volatile int *abort_flag = &ctl->abort_flag;
    // TMEM: O [0, DV) | S1 buffers [DV, DV+128) | S2 buffers [DV+128, DV+256)
    const uint32_t tS1_0 = DV, tS2_0 = DV + 2 * kBN2;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (elect_one()) {
            tma_prefetch_desc(&tmQ1);
            tma_prefetch_desc(&tmK1);
            tma_prefetch_desc(&tmQ2);
            tma_prefetch_desc(&tmK2);
            tma_prefetch_desc(&tmV);
            uint32_t kt = 0, vt = 0;
            int nq = 0;
            bool ok = true;
            Item2 it;
            for (int r = 0; ok && item2_of(p, p.hs, r, G, cid, it); ++r) {
                const int h = it.head, g = h / r_grp;
                if (r > 0 && !wait_quick(&ctl->q_empty, (r - 1) & 1, p.err, abort_flag)) break;
                mbar_arrive_expect_tx(&ctl->q_full, 2 * LY::Q_BYTES);
#pragma unroll
                for (int blk = 0; blk < D / 64; ++blk) {
                    tma_load_4d(smem + LY::OFF_Q1 + blk * kBM * 128, &tmQ1, &ctl->q_full, blk * 64, h, it.q0, it.b);
                    tma_load_4d(smem + LY::OFF_Q2 + blk * kBM * 128, &tmQ2, &ctl->q_full, blk * 64, g, it.q0, it.b);
                }
                ++nq;
                auto load_k = [&](int j) -> bool {
                    const uint32_t gk = kt + j;
                    const int st = gk % KS;
                    if (gk >= KS && !wait_quick(&ctl->k_empty[st], ((gk / KS) - 1) & 1, p.err, abort_flag))
                        return false;
                    uint8_t *sb = smem + LY::OFF_K + st * LY::KST_BYTES;
                    mbar_arrive_expect_tx(&ctl->k_full[st], LY::KST_BYTES);
#pragma unroll
                    for (int blk = 0; blk < D / 64; ++blk) {
                        tma_load_4d(sb + blk * kBN2 * 128, &tmK1, &ctl->k_full[st], blk * 64, h, j * kBN2, it.b);
                        tma_load_4d(sb + LY::K_BYTES + blk * kBN2 * 128, &tmK2, &ctl->k_full[st], blk * 64, g,
                                    j * kBN2, it.b);
                    }
                    return true;
                };
                auto load_v = [&](int j) -> bool {
                    const uint32_t gv = vt + j;
                    const int st = gv % VS;
                    if (gv >= VS && !wait_quick(&ctl->v_empty[st], ((gv / VS) - 1) & 1, p.err, abort_flag))
                        return false;
                    uint8_t *sb = smem + LY::OFF_V + st * LY::V_BYTES;
                    mbar_arrive_expect_tx(&ctl->v_full[st], LY::V_BYTES);
#pragma unroll
                    for (int blk = 0; blk < DV / 64; ++blk)
                        tma_load_4d(sb + blk * kBN2 * 128, &tmV, &ctl->v_full[st], blk * 64, h, j * kBN2, it.b);
                    return true;
                };
                // K runs two tiles ahead of V (QK(j+2) is issued right after PV(j))
                int kdone = 0, vdone = 0;
                for (int t = 0; ok && t < 2 && t < it.nkv; ++t) {
                    ok = load_k(t);
                    if (ok) ++kdone;
                }
                for (int j = 0; ok && j < it.nkv; ++j) {
                    if (j + 2 < it.nkv) {
                        ok = load_k(j + 2);
                        if (!ok) break;
                        ++kdone;
                    }
                    ok = load_v(j);
                    if (ok) ++vdone;
                }
                kt += kdone;
                vt += vdone;
            }
            if (nq > 0) drain_wait(&ctl->q_full, (nq - 1) & 1, p.err);
            for (uint32_t j = (kt > KS ? kt - KS : 0); j < kt; ++j)
                drain_wait(&ctl->k_full[j % KS], (j / KS) & 1, p.err);
            for (uint32_t j = (vt > VS ? vt - VS : 0); j < vt; ++j)
                drain_wait(&ctl->v_full[j % VS], (j / VS) & 1, p.err);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (elect_one()) {
            const uint32_t q1a = smem_u32(smem + LY::OFF_Q1);
            const uint32_t q2a = smem_u32(smem + LY::OFF_Q2);
            const uint32_t k0a = smem_u32(smem + LY::OFF_K);
            const uint32_t v0a = smem_u32(smem + LY::OFF_V);
            uint32_t kt = 0, vt = 0, gt = 0;
            bool ok = true;
            Item2 it;
            for (int r = 0; ok && item2_of(p, p.hs, r, G, cid, it); ++r) {
                const int nkv = it.nkv;
                if (!wait_quick(&ctl->q_full, r & 1, p.err, abort_flag)) break;
                // logits of the first two tiles (overlaps the previous epilogue)
                for (int t = 0; t < 2 && t < nkv; ++t) {
                    const uint32_t gk = kt + t, gs = gt + t;
                    if (!wait_quick(&ctl->k_full[gk % KS], (gk / KS) & 1, p.err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ka = k0a + (gk % KS) * LY::KST_BYTES;
                    issue_qk<D, kBN2>(tmem + tS1_0 + (gs & 1) * kBN2, q1a, ka);
                    issue_qk<D, kBN2>(tmem + tS2_0 + (gs & 1) * kBN2, q2a, ka + LY::K_BYTES);
                    mma_commit(&ctl->s_full[gs & 1]);
                    mma_commit(&ctl->k_empty[gk % KS]);
                }
                if (!ok) break;
                if (nkv <= 2) mma_commit(&ctl->q_empty);
                if (r > 0 && !wait_quick(&ctl->o_free, (r - 1) & 1, p.err, abort_flag)) break;
                for (int j = 0; j < nkv; ++j) {
                    const uint32_t gs = gt + j, gv = vt + j;
                    const int bb = gs & 1;
                    if (!wait_quick(&ctl->p_full[bb], (gs >> 1) & 1, p.err, abort_flag)) { ok = false; break; }
                    if (!wait_quick(&ctl->v_full[gv % VS], (gv / VS) & 1, p.err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    issue_pv_split<DV>(tmem, tmem + tS1_0 + bb * kBN2, v0a + (gv % VS) * LY::V_BYTES, j > 0);
                    mma_commit(&ctl->v_empty[gv % VS]);
                    const int jn = j + 2;
                    if (jn < nkv) {
                        const uint32_t gk = kt + jn;
                        if (!wait_quick(&ctl->k_full[gk % KS], (gk / KS) & 1, p.err, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t ka = k0a + (gk % KS) * LY::KST_BYTES;
                        issue_qk<D, kBN2>(tmem + tS1_0 + bb * kBN2, q1a, ka);
                        issue_qk<D, kBN2>(tmem + tS2_0 + bb * kBN2, q2a, ka + LY::K_BYTES);
                        mma_commit(&ctl->s_full[bb]);
                        mma_commit(&ctl->k_empty[gk % KS]);
                        if (jn == nkv - 1) mma_commit(&ctl->q_empty);
                    }
                }
                if (!ok) break;
                mma_commit(&ctl->o_final);
                kt += nkv;
                vt += nkv;
                gt += nkv;
            }
            mma_commit(&ctl->mma_idle);
            drain_wait(&ctl->mma_idle, 0, p.err);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ difference map + epilogue
        const int half = (warp - 2) / 4;
        const int quarter = warp % 4;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        const int heads = p.hs + p.hn;
        uint32_t gt = 0;
        Item2 it;
        for (int r = 0; item2_of(p, p.hs, r, G, cid, it); ++r) {
            const int h = it.head, g = h / r_grp;
            const int qrow = it.q0 + row;
            const bool in = qrow < p.L;
            const int last_key = p.causal ? min(p.koff + qrow, p.Lk - 1) : p.Lk - 1;
            const float lam = p.lambda[h];
            // rows past L get lse = +inf, so every P of theirs is 0
            const float neg1 = in ? -p.lse[(static_cast<size_t>(it.b) * heads + h) * p.lse_ld + qrow] : -INFINITY;
            const float neg2 = in ? -p.lse[(static_cast<size_t>(it.b) * heads + p.hs + g) * p.lse_ld + qrow] : -INFINITY;
            const float nlam = -lam;
            bool ok = true;
            for (int j = 0; j < it.nkv; ++j) {
                const uint32_t gs = gt + j;
                const int bb = gs & 1;
                // per-lane wait: a failed one sets the error word and the flag that ends every
                // later wait at once; the loop runs on, so the barrier counts stay whole
                if (!wait_quick(&ctl->s_full[bb], (gs >> 1) & 1, p.err, abort_flag)) ok = false;
                tc_fence_after();
                const uint32_t tS1 = tmem + lane_off + tS1_0 + bb * kBN2 + half * 32;
                const uint32_t tS2 = tmem + lane_off + tS2_0 + bb * kBN2 + half * 32;
                uint32_t r1[32], r2[32];
                tmem_ld32(tS1, r1);
                tmem_ld32(tS2, r2);
                tmem_ld_wait_regs(r1);
                reg_fence(r2);
                const int k0 = j * kBN2 + half * 32;
                uint32_t pk[16];
                auto probs = [&](auto masked) {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float x0 = __uint_as_float(r1[e]), x1 = __uint_as_float(r1[e + 1]);
                        float y0 = __uint_as_float(r2[e]), y1 = __uint_as_float(r2[e + 1]);
                        ffma2(x0, x1, sl2, sl2, neg1, neg1);
                        ffma2(y0, y1, sl2, sl2, neg2, neg2);
                        float p0 = fmaf(nlam, fast_exp2(y0), fast_exp2(x0));
                        float p1 = fmaf(nlam, fast_exp2(y1), fast_exp2(x1));
                        if constexpr (decltype(masked)::value) {
                            if (k0 + e > last_key) p0 = 0.f;
                            if (k0 + e + 1 > last_key) p1 = 0.f;
                        }
                        pk[e / 2] = pack_bf16x2(p0, p1);
                    }
                };
                // the per-key test only where some row of the warp has keys past its last one
                if (__any_sync(0xffffffffu, k0 + 31 > last_key))
                    probs(std::true_type{});
                else
                    probs(std::false_type{});
                tmem_st16(tS1, pk);                  // over the S1 columns this half read
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&ctl->p_full[bb]);
            }
            tmem_ld_wait();

            // ------------------------------------------------ epilogue: headwise norm
            ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
            if (ok) ok = warp_wait(&ctl->o_final, r & 1, p.err, abort_flag);
            tc_fence_after();
            constexpr int HC = DV / 2;               // this half's output columns
            const uint32_t tO = tmem + lane_off + half * HC;
            float ss = 0.f;
            if (ok) {
#pragma unroll
                for (int cc = 0; cc < HC / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + cc * 32, o);
                    tmem_ld_wait_regs(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) ss = fmaf(__uint_as_float(o[e]), __uint_as_float(o[e]), ss);
                }
            }
            ctl->ss_part[half][row] = ss;
            named_bar_sync(1, kSmThreads);
            const float ss_tot = ctl->ss_part[0][row] + ctl->ss_part[1][row];
            ok = __all_sync(0xffffffffu, ok);
            const float yscale =
                p.no_norm ? 1.f : (1.f - p.lambda_init) * rsqrtf(ss_tot / static_cast<float>(DV) + p.eps);
            if (ok) {
                __nv_bfloat16 *orow = p.out + ((static_cast<size_t>(it.b) * p.L + qrow) * p.hs + h) * DV + half * HC;
#pragma unroll
                for (int cc = 0; cc < HC / 32; ++cc) {
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
            // the accumulator may now be overwritten by the next item's first PV;
            // ss_part is read before the next item's barrier lets anyone rewrite it
            tc_fence_before();
            mbar_arrive(&ctl->o_free);
            gt += it.nkv;
            if (bar_red_or(1, kSmThreads, !ok || *abort_flag)) break;
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

int sm_count(int *sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

void fill_params(P2Params &p, const PrefillArgs &a, float *lse, int lse_ld) {
    p.lambda = a.lambda;
    p.lse = lse;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.err = a.dev_err;
    p.lambda_init = a.lambda_init;
    p.eps = a.eps;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.d)));
    p.B = a.B;
    p.L = a.L;
    p.hs = a.hs;
    p.hn = a.hn;
    p.dv = a.dv;
    p.causal = a.causal;
    p.nqt = (a.L + kBM - 1) / kBM;
    p.no_norm = (a.flags & GDA_FLAG_NO_NORM) ? 1 : 0;
    p.lse_ld = lse_ld;
    p.Lk = a.Lk > 0 ? a.Lk : a.L;
    p.koff = p.Lk - a.L;
}

// Queries: L rows per sequence; keys (and values): Lk rows.
bool qk_maps(const PrefillArgs &a, CUtensorMap *mQ1, CUtensorMap *mK1, CUtensorMap *mQ2, CUtensorMap *mK2) {
    const uint64_t B = a.B, L = a.L, Lk = a.Lk > 0 ? a.Lk : a.L, hs = a.hs, hn = a.hn, d = a.d;
    const uint32_t boxq[4] = {64, 1, kBM, 1}, boxk[4] = {64, 1, kBN2, 1};
    {
        const uint64_t dq[4] = {d, hs, L, B}, dk[4] = {d, hs, Lk, B};
        const uint64_t sq[3] = {d * 2, hs * d * 2, L * hs * d * 2}, sk[3] = {d * 2, hs * d * 2, Lk * hs * d * 2};
        if (!encode_tmap_4d_bf16(mQ1, a.q1, dq, sq, boxq)) return false;
        if (!encode_tmap_4d_bf16(mK1, a.k1, dk, sk, boxk)) return false;
    }
    const uint64_t dq[4] = {d, hn, L, B}, dk[4] = {d, hn, Lk, B};
    const uint64_t sq[3] = {d * 2, hn * d * 2, L * hn * d * 2}, sk[3] = {d * 2, hn * d * 2, Lk * hn * d * 2};
    if (!encode_tmap_4d_bf16(mQ2, a.q2, dq, sq, boxq)) return false;
    return encode_tmap_4d_bf16(mK2, a.k2, dk, sk, boxk);
}

template <int D>
int launch_lse_impl(const PrefillArgs &a, const CUtensorMap &mQ1, const CUtensorMap &mK1, const CUtensorMap &mQ2,
                    const CUtensorMap &mK2, const P2Params &p, int sms, cudaStream_t stream) {
    const long long items1 = static_cast<long long>(p.nqt) * a.B * (a.hs + a.hn);
    if (items1 > 0x7fffffffLL) return GDA_ERR_UNSUPPORTED;
    auto k1 = gda_lse_tc_kernel<D>;
    constexpr int smem1 = lse_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, smem1);
    if (e != cudaSuccess) return record_cuda_error(e);
    long long g1 = 2LL * sms;                // two CTAs per SM
    if (g1 > items1) g1 = items1;
    k1<<<static_cast<unsigned>(g1), kThreads2, smem1, stream>>>(mQ1, mK1, mQ2, mK2, p);
    e = cudaGetLastError();
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

template <int D, int DV>
int launch_2pass_impl(const PrefillArgs &a, float *lse, cudaStream_t stream) {
    CUtensorMap mQ1, mK1, mQ2, mK2, mV;
    const uint64_t B = a.B, Lk = a.Lk > 0 ? a.Lk : a.L, hs = a.hs, dv = a.dv;
    if (!qk_maps(a, &mQ1, &mK1, &mQ2, &mK2)) return GDA_ERR_CUDA;
    {
        const uint64_t dims[4] = {dv, hs, Lk, B};
        const uint64_t str[3] = {dv * 2, hs * dv * 2, Lk * hs * dv * 2};
        const uint32_t box[4] = {64, 1, kBN2, 1};
        if (!encode_tmap_4d_bf16(&mV, a.v, dims, str, box)) return GDA_ERR_CUDA;
    }
    P2Params p;
    fill_params(p, a, lse, a.L);
    int sms = 0;
    int st = sm_count(&sms);
    if (st != GDA_OK) return st;
    st = launch_lse_impl<D>(a, mQ1, mK1, mQ2, mK2, p, sms, stream);
    if (st != GDA_OK) return st;
    const long long items2 = static_cast<long long>(p.nqt) * a.B * a.hs;

    auto k2 = gda_diffmap_tc_kernel<D, DV>;
    constexpr int smem2 = dm_smem_bytes<D, DV>();
    static_assert(smem2 <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2);
    if (e != cudaSuccess) return record_cuda_error(e);
    long long g2 = sms;
    if (g2 > items2) g2 = items2;
    k2<<<static_cast<unsigned>(g2), kThreads2, smem2, stream>>>(mQ1, mK1, mQ2, mK2, mV, p);
    e = cudaGetLastError();
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

}  // namespace

size_t prefill_2pass_workspace_bytes(int B, int L, int hs, int hn) {
    return sizeof(float) * static_cast<size_t>(B) * static_cast<size_t>(hs + hn) * static_cast<size_t>(L);
}

int launch_lse_pass(const PrefillArgs &a, float *lse, int lse_ld, cudaStream_t stream) {
    CUtensorMap mQ1, mK1, mQ2, mK2;
    if (!qk_maps(a, &mQ1, &mK1, &mQ2, &mK2)) return GDA_ERR_CUDA;
    P2Params p;
    fill_params(p, a, lse, lse_ld);
    int sms = 0;
    const int st = sm_count(&sms);
    if (st != GDA_OK) return st;
    if (a.d == 64) return launch_lse_impl<64>(a, mQ1, mK1, mQ2, mK2, p, sms, stream);
    if (a.d == 128) return launch_lse_impl<128>(a, mQ1, mK1, mQ2, mK2, p, sms, stream);
    return GDA_ERR_UNSUPPORTED;
}

int launch_prefill_2pass(const PrefillArgs &a, void *workspace, cudaStream_t stream) {
    float *lse = static_cast<float *>(workspace);
    if (a.d == 64 && a.dv == 128) return launch_2pass_impl<64, 128>(a, lse, stream);
    if (a.d == 64 && a.dv == 256) return launch_2pass_impl<64, 256>(a, lse, stream);
    if (a.d == 128 && a.dv == 128) return launch_2pass_impl<128, 128>(a, lse, stream);
    if (a.d == 128 && a.dv == 256) return launch_2pass_impl<128, 256>(a, lse, stream);
    return GDA_ERR_UNSUPPORTED;
}

}  // namespace gda
