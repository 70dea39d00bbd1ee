// Causal (or full) grouped differential attention prefill for sm_103a:
// TMA-staged bf16 tiles, tcgen05 MMAs accumulating in TMEM, two online
// softmax states and the fused difference + headwise RMSNorm epilogue.
//
// What it computes: for signal head h with noise head g = h / (h_s / h_n),
//   o = softmax(Q1_h K1_h^T / sqrt d) V_h - lambda_h softmax(Q2_g K2_g^T / sqrt d) V_h
//   y = (1 - lambda_init) o / sqrt(mean(o^2) + eps)
// ("Differential Attention in Large Language Models ...", sections
// "Differential Attention Architecture" and "Headwise Normalization";
// noise-head sharing from the "Grouped Differential Attention" abstract).
// Both maps are normalised before the subtraction, so the kernel carries two
// running (max, sum) states and two float32 accumulators per query row; no
// L x L map ever leaves the SM.
//
// Persistent: one CTA per SM (a CTA pair per two SMs for dv = 256) walks a
// list of work items (query tile of 128 rows, batch b, signal head h; the
// pair splits dv into two 128-column slices).  Barriers and TMEM are set up
// once; the next item's Q load and first two QK MMAs overlap the current
// item's epilogue.
// 10 warps:
//   warp 0       TMA producer (one elected lane): Q1/Q2 once, then a ring of
//                K stages (K1 and K2 tiles) and a ring of V stages;
//   warp 1       TMEM allocator and MMA issuer (one elected lane);
//   warps 2-5    softmax of the signal map, warps 6-9 of the noise map
//                (thread = query row = TMEM lane).  The next S tile's row is
//                requested from TMEM as soon as the current row's exponentials
//                are done, so its latency overlaps the P-store wait and the
//                barrier arrive.
// KV tiles are 64 keys.  TMEM (512 columns): O1 [0,128) | O2 [128,256) |
// S1 tiles [256,320) [320,384) | S2 tiles [384,448) [448,512): each map's S
// is double-buffered, so QK(j+2) runs on the tensor core while the softmax
// of tile j+1 runs, and the softmax warps never wait on their own map's PV.
// P overwrites the first 32 columns of its S tile and feeds the PV MMA
// straight from TMEM.  A row's reference maximum is taken exactly on its
// first key tile only; later tiles exponentiate against it directly (no
// per-tile maximum on the critical path) and only a tile whose sum of P
// grows past 2^16 is redone with its exact maximum, rescaling the row's sum
// and accumulator.
// dv = 256 is split over a 2-CTA cluster; the two CTAs exchange the per-row
// sum of squares through distributed shared memory (remote store plus remote
// mbarrier arrive) for the RMSNorm.
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

constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = 32 * (2 + kSoftmaxWarps);
constexpr float kSumLimit = 65536.0f;       // per-tile P sum that triggers a new reference

template <int D> struct TcCfg;
template <> struct TcCfg<64> { static constexpr int BN = 64, KS = 4, VS = 4; };
template <> struct TcCfg<128> { static constexpr int BN = 64, KS = 3, VS = 3; };

struct Ctrl {
    uint64_t q_full, q_empty;
    uint64_t k_full[4], k_empty[4];
    uint64_t v_full[4], v_empty[4];
    uint64_t s_full[2][2];      // [map][S buffer]
    uint64_t p_full[2][2];      // [map][S buffer]
    uint64_t o_done[2];         // [map]: one phase per PV
    uint64_t o_final;           // every MMA of the current item has completed
    uint64_t o_free;            // the epilogue has read the accumulators
    uint64_t peer_bar[2];       // peer CTA's sum of squares arrived (dv = 256)
    uint64_t mma_idle;
    uint32_t tmem_base;
    int abort_flag;
    float l_row[2][kBM];        // [map][row]
    float ss_part[2][kBM];      // [warpgroup][row]
    float ss_peer[2][kBM];
};

template <int D> struct Layout {
    static constexpr int BN = TcCfg<D>::BN;
    static constexpr int KS = TcCfg<D>::KS;
    static constexpr int VS = TcCfg<D>::VS;
    static constexpr int Q_BYTES = kBM * D * 2;
    static constexpr int K_BYTES = BN * D * 2;          // one of K1 / K2
    static constexpr int KST_BYTES = 2 * K_BYTES;       // K stage: K1 then K2
    static constexpr int V_BYTES = BN * kDVS * 2;       // V stage
    static constexpr int OFF_Q1 = 0;
    static constexpr int OFF_Q2 = Q_BYTES;
    static constexpr int OFF_K = 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KS * KST_BYTES;
    static constexpr int OFF_OUT = OFF_V + VS * V_BYTES;
    // output staging for TMA stores: 32 rows x 64 columns (128-byte
    // swizzle) per softmax warp, where shared memory allows (d = 64)
    static constexpr bool TMA_OUT = D == 64;
    static constexpr int OUT_BYTES = TMA_OUT ? kSoftmaxWarps * 32 * 128 : 0;
    static constexpr int TILES = OFF_OUT + OUT_BYTES;
    static constexpr int TOTAL = TILES + (int)((sizeof(Ctrl) + 1023) / 1024) * 1024 + 1024;
    static_assert(TOTAL <= 232448, "shared memory budget");
    static_assert(256 + 4 * BN <= 512, "TMEM budget");
    static_assert(KS <= 4 && VS <= 4, "barrier arrays");
};

struct TcParams {
    const float *lambda;
    __nv_bfloat16 *out;
    unsigned *err;
    float lambda_init, eps, scale_log2;
    int B, L, hs, hn, dv, causal, nslices, nqt, no_norm;
    int Lk, koff;      // keys per sequence; query row i sits at key position koff + i (koff = Lk - L)
};

// Work item = (query tile, batch, signal head); item 0 is the longest (last
// query tile).  Persistent CTAs (or CTA pairs for dv = 256) take items in a
// snake order: round r takes item r*G + c for even r and r*G + G-1-c for odd
// r (G CTAs or pairs, c this CTA's index), which evens out the causal lengths.
struct Item {
    int b, h, g, q0, nkv;
};

__device__ __forceinline__ bool item_of(const TcParams &p, int r, int G, int cid, int bn, Item &it) {
    const int nitems = p.nqt * p.B * p.hs;
    const int k = (r & 1) ? (G - 1 - cid) : cid;
    const long long idx = static_cast<long long>(r) * G + k;
    if (idx >= nitems) return false;
    const int i = static_cast<int>(idx);
    const int qt = p.nqt - 1 - i / (p.B * p.hs);
    const int rem = i % (p.B * p.hs);
    it.b = rem / p.hs;
    it.h = rem % p.hs;
    it.g = it.h / (p.hs / p.hn);
    it.q0 = qt * kBM;
    const int kv_end = p.causal ? min(p.Lk, p.koff + it.q0 + kBM) : p.Lk;
    it.nkv = (kv_end + bn - 1) / bn;
    return true;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
gda_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ1,
                      const __grid_constant__ CUtensorMap tmK1,
                      const __grid_constant__ CUtensorMap tmQ2,
                      const __grid_constant__ CUtensorMap tmK2,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmO, const TcParams p) {
    using LY = Layout<D>;
    constexpr int BN = LY::BN;
    constexpr int KS = LY::KS;
    constexpr int VS = LY::VS;

    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, offset from the shared array itself so that accesses stay in the
    // shared state space (32-bit addresses)
    uint8_t *smem = smem_raw + ((0u - smem_u32(smem_raw)) & 1023u);
    Ctrl *ctl = reinterpret_cast<Ctrl *>(smem + LY::TILES);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int slice = blockIdx.x % p.nslices;
    const int cid = blockIdx.x / p.nslices;
    const int G = gridDim.x / p.nslices;

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
        for (int m = 0; m < 2; ++m) {
            for (int bb = 0; bb < 2; ++bb) {
                mbar_init(&ctl->s_full[m][bb], 1);
                mbar_init(&ctl->p_full[m][bb], 128);
            }
            mbar_init(&ctl->o_done[m], 1);
            mbar_init(&ctl->peer_bar[m], 128);
        }
        mbar_init(&ctl->o_final, 1);
        mbar_init(&ctl->o_free, 32 * kSoftmaxWarps);
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
    if (p.nslices == 2) cluster_sync_all();   // peer CTA is running before any DSMEM access
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;

    if (warp == 0) {
        // ================================================= TMA producer
        if (elect_one()) {
            tma_prefetch_desc(&tmQ1);
            tma_prefetch_desc(&tmK1);
            tma_prefetch_desc(&tmQ2);
            tma_prefetch_desc(&tmK2);
            tma_prefetch_desc(&tmV);
            uint32_t kt = 0, vt = 0;           // K / V tiles issued so far (all items)
            int nq = 0;                        // Q loads issued
            bool ok = true;
            Item it;
            for (int r = 0; ok && item_of(p, r, G, cid, BN, it); ++r) {
                // Q of the previous item must have been read by its last QK
                if (r > 0 && !wait_quick(&ctl->q_empty, (r - 1) & 1, p.err, abort_flag)) break;
                mbar_arrive_expect_tx(&ctl->q_full, 2 * LY::Q_BYTES);
#pragma unroll
                for (int blk = 0; blk < D / 64; ++blk) {
                    tma_load_4d(smem + LY::OFF_Q1 + blk * kBM * 128, &tmQ1, &ctl->q_full, blk * 64, it.h,
                                it.q0, it.b);
                    tma_load_4d(smem + LY::OFF_Q2 + blk * kBM * 128, &tmQ2, &ctl->q_full, blk * 64, it.g,
                                it.q0, it.b);
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
                        tma_load_4d(sb + blk * BN * 128, &tmK1, &ctl->k_full[st], blk * 64, it.h, j * BN, it.b);
                        tma_load_4d(sb + LY::K_BYTES + blk * BN * 128, &tmK2, &ctl->k_full[st], blk * 64, it.g,
                                    j * BN, it.b);
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
                    for (int blk = 0; blk < kDVS / 64; ++blk)
                        tma_load_4d(sb + blk * BN * 128, &tmV, &ctl->v_full[st], slice * kDVS + blk * 64, it.h,
                                    j * BN, it.b);
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
            const uint32_t tO1 = tmem, tO2 = tmem + 128;
            const uint32_t tS1 = tmem + 256, tS2 = tmem + 256 + 2 * BN;   // + buffer * BN
            const uint32_t q1a = smem_u32(smem + LY::OFF_Q1);
            const uint32_t q2a = smem_u32(smem + LY::OFF_Q2);
            const uint32_t k0a = smem_u32(smem + LY::OFF_K);
            const uint32_t v0a = smem_u32(smem + LY::OFF_V);
            uint32_t kt = 0, vt = 0, gt = 0;
            bool ok = true;
            Item it;
            for (int r = 0; ok && item_of(p, r, G, cid, BN, it); ++r) {
                const int nkv = it.nkv;
                if (!wait_quick(&ctl->q_full, r & 1, p.err, abort_flag)) break;
                // QK of the item's first two tiles; their S buffers were last
                // read by PVs already issued.  This overlaps the previous
                // item's epilogue.
                for (int t = 0; t < 2 && t < nkv; ++t) {
                    const uint32_t gk = kt + t, gs = gt + t;
                    if (!wait_quick(&ctl->k_full[gk % KS], (gk / KS) & 1, p.err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ka = k0a + (gk % KS) * LY::KST_BYTES;
                    issue_qk<D, BN>(tS1 + (gs & 1) * BN, q1a, ka);
                    mma_commit(&ctl->s_full[0][gs & 1]);
                    issue_qk<D, BN>(tS2 + (gs & 1) * BN, q2a, ka + LY::K_BYTES);
                    mma_commit(&ctl->s_full[1][gs & 1]);
                    mma_commit(&ctl->k_empty[gk % KS]);
                }
                if (!ok) break;
                if (nkv <= 2) mma_commit(&ctl->q_empty);
                // the accumulators are free once the previous item's epilogue has read them
                if (r > 0 && !wait_quick(&ctl->o_free, (r - 1) & 1, p.err, abort_flag)) break;
                for (int j = 0; j < nkv; ++j) {
                    const uint32_t gs = gt + j, gv = vt + j;
                    const int bb = gs & 1;
                    const uint32_t va = v0a + (gv % VS) * LY::V_BYTES;
                    const int jn = j + 2;                       // next tile for this S buffer
                    const bool more = jn < nkv;
                    const uint32_t gk = kt + jn;
                    const uint32_t kan = k0a + (gk % KS) * LY::KST_BYTES;
                    // signal map: PV1(j), then QK1(j+2) into the S1 buffer PV1(j) just read
                    if (!wait_quick(&ctl->p_full[0][bb], (gs >> 1) & 1, p.err, abort_flag)) { ok = false; break; }
                    if (!wait_quick(&ctl->v_full[gv % VS], (gv / VS) & 1, p.err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    issue_pv<BN>(tO1, tS1 + bb * BN, va, j > 0);
                    mma_commit(&ctl->o_done[0]);
                    if (more) {
                        if (!wait_quick(&ctl->k_full[gk % KS], (gk / KS) & 1, p.err, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        issue_qk<D, BN>(tS1 + bb * BN, q1a, kan);
                        mma_commit(&ctl->s_full[0][bb]);
                    }
                    // noise map: PV2(j), release V(j), then QK2(j+2) and release K(j+2)
                    if (!wait_quick(&ctl->p_full[1][bb], (gs >> 1) & 1, p.err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    issue_pv<BN>(tO2, tS2 + bb * BN, va, j > 0);
                    mma_commit(&ctl->o_done[1]);
                    mma_commit(&ctl->v_empty[gv % VS]);
                    if (more) {
                        issue_qk<D, BN>(tS2 + bb * BN, q2a, kan + LY::K_BYTES);
                        mma_commit(&ctl->s_full[1][bb]);
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
            // every issued MMA completes before TMEM is released
            mma_commit(&ctl->mma_idle);
            drain_wait(&ctl->mma_idle, 0, p.err);
        }
        __syncwarp();
    } else {
        // ================================================= softmax groups
        const int m = (warp - 2) / 4;             // 0: signal map, 1: noise map
        const int quarter = warp % 4;             // TMEM lanes this warp may touch
        const int row = quarter * 32 + lane;      // query row in the tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tSm = tmem + 256 + m * 2 * BN + lane_off;   // + buffer * BN
        const uint32_t tOm = tmem + m * 128 + lane_off;
        const float sl2 = p.scale_log2;
        uint32_t gt = 0;
        Item it;
        for (int r = 0; item_of(p, r, G, cid, BN, it); ++r) {
            const int nkv = it.nkv;
            const int qrow = it.q0 + row;
            const int last_key = p.causal ? min(p.koff + qrow, p.Lk - 1) : p.Lk - 1;
            const float lam = p.lambda[it.h];     // loaded now, used by the epilogue
            float m_ref = -INFINITY;
            float l = 0.f;
            bool ok = true;

            // r holds the current tile's S row; the next tile's row is requested
            // into the same registers once the exponentials have consumed them,
            // so its TMEM latency overlaps the P-store wait and the barrier arrive.
            uint32_t rr[BN];
            if (warp_wait(&ctl->s_full[m][gt & 1], (gt >> 1) & 1, p.err, abort_flag)) {
                tc_fence_after();
#pragma unroll
                for (int cch = 0; cch < BN / 32; ++cch)
                    tmem_ld32(tSm + (gt & 1) * BN + cch * 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[cch * 32]));
                tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&rr[0]));
                reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&rr[32]));
            } else {
                ok = false;
            }
            for (int j = 0; ok && j < nkv; ++j) {
                const uint32_t gs = gt + j;
                const uint32_t tS = tSm + (gs & 1) * BN;
                const int k0 = j * BN;
                const bool need_mask = (p.causal && k0 + BN - 1 > p.koff + it.q0) || (k0 + BN > p.Lk);
                if (need_mask) {
#pragma unroll
                    for (int e = 0; e < BN; ++e)
                        if (k0 + e > last_key) rr[e] = __float_as_uint(-INFINITY);
                }
                // exact row maximum of the tile (exp2 units)
                auto row_max = [&]() -> float {
                    float mx4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx4[i] = __uint_as_float(rr[i]);
#pragma unroll
                    for (int e = 4; e + 8 <= BN; e += 8)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            mx4[i] = max3f(mx4[i], __uint_as_float(rr[e + 2 * i]), __uint_as_float(rr[e + 2 * i + 1]));
                    float mx = max3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
#pragma unroll
                    for (int e = 4 + ((BN - 4) / 8) * 8; e < BN; ++e) mx = fmaxf(mx, __uint_as_float(rr[e]));
                    return mx * sl2;
                };
                // P = 2^(s*scale - m) stored packed over S (hidden keys hold
                // -inf and give 0); returns the tile's sum of P
                auto exp_store = [&](float m) -> float {
                    const float neg_m = -m;
                    float sa = 0.f, sb = 0.f, sc = 0.f, sd = 0.f;
#pragma unroll
                    for (int hh = 0; hh < BN / 32; ++hh) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            float x0 = __uint_as_float(rr[hh * 32 + e]), x1 = __uint_as_float(rr[hh * 32 + e + 1]);
                            float x2 = __uint_as_float(rr[hh * 32 + e + 2]), x3 = __uint_as_float(rr[hh * 32 + e + 3]);
                            ffma2(x0, x1, sl2, sl2, neg_m, neg_m);
                            ffma2(x2, x3, sl2, sl2, neg_m, neg_m);
                            x0 = fast_exp2(x0);
                            x1 = fast_exp2(x1);
                            x2 = fast_exp2(x2);
                            x3 = fast_exp2(x3);
                            fadd2(sa, sb, x0, x1);
                            fadd2(sc, sd, x2, x3);
                            pk[e / 2] = pack_bf16x2(x0, x1);
                            pk[e / 2 + 1] = pack_bf16x2(x2, x3);
                        }
                        tmem_st16(tS + hh * 16, pk);
                    }
                    return (sa + sb) + (sc + sd);
                };
                // The reference m_ref is the exact maximum of the first tile.
                // Later tiles reuse it: floating point keeps P's relative
                // precision at any scale, so m_ref only has to keep P and the
                // sums far from overflow.  A tile whose P sum exceeds
                // kSumLimit (some P > kSumLimit / BN, or inf) is redone with
                // its exact maximum as the new reference, and the row's sum
                // and accumulator are rescaled.
                if (j == 0) m_ref = row_max();
                float alpha = 1.f;
                bool rescale = false;
                float tsum = exp_store(m_ref);
                if (__any_sync(0xffffffffu, !(tsum <= kSumLimit))) {
                    if (!(tsum <= kSumLimit)) {
                        const float mt = row_max();
                        if (mt > m_ref) {
                            alpha = fast_exp2(m_ref - mt);
                            m_ref = mt;
                            rescale = true;
                        }
                    }
                    tmem_st_wait();            // the first P store lands before it is overwritten
                    tsum = exp_store(m_ref);   // every lane again: the TMEM store is warp-wide
                }
                l = l * alpha + tsum;
                // request the next S tile into rr
                const bool more = j + 1 < nkv;
                if (more) {
                    if (!warp_wait(&ctl->s_full[m][(gs + 1) & 1], ((gs + 1) >> 1) & 1, p.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tSn = tSm + ((gs + 1) & 1) * BN;
#pragma unroll
                    for (int cch = 0; cch < BN / 32; ++cch)
                        tmem_ld32(tSn + cch * 32, *reinterpret_cast<uint32_t(*)[32]>(&rr[cch * 32]));
                }
                tmem_st_wait();
                if (__any_sync(0xffffffffu, rescale)) {
                    // the accumulator may only be touched once PV(j-1) has completed
                    if (!warp_wait(&ctl->o_done[m], (gs - 1) & 1, p.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int cch = 0; cch < kDVS / 32; ++cch) {
                        uint32_t o[32];
                        tmem_ld32(tOm + cch * 32, o);
                        tmem_ld_wait_regs(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tOm + cch * 32, o);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(&ctl->p_full[m][gs & 1]);
                if (more) {
                    tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&rr[0]));
                    reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&rr[32]));
                }
            }
            // drain any TMEM load still in flight after an early exit
            tmem_ld_wait();

            // ------------------------------------------------ epilogue of the item
            // A row's two halves (map 0's warp: columns 0-63 of O1 and O2, map
            // 1's warp: columns 64-127) sit in the two warps of one lane
            // quarter; only those two warps exchange the row sums and the sums
            // of squares, on a named barrier of their own, so a pair never
            // waits for the other quarters.
            const uint32_t pair_bar = 2 + quarter;
            ctl->l_row[m][row] = l;
            named_bar_sync(pair_bar, 64);
            const float l1 = ctl->l_row[0][row];
            const float l2 = ctl->l_row[1][row];
            ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
            if (ok) ok = warp_wait(&ctl->o_final, r & 1, p.err, abort_flag);
            tc_fence_after();
            const float inv1 = 1.f / l1;
            const float c2 = lam / l2;
            const uint32_t tO1 = tmem + lane_off, tO2 = tmem + 128 + lane_off;
            const int col0 = m * 64;                  // this warpgroup's 64 columns of the slice
            float ss = 0.f;
            if (ok) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t r1[32], r2[32];
                    tmem_ld32(tO1 + col0 + cc * 32, r1);
                    tmem_ld32(tO2 + col0 + cc * 32, r2);
                    tmem_ld_wait_regs(r1);
                    reg_fence(r2);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        // both products rounded before the subtraction (no FMA
                        // contraction), so equal maps with lambda = 1 cancel exactly
                        const float o = __fmul_rn(__uint_as_float(r1[e]), inv1) - __fmul_rn(__uint_as_float(r2[e]), c2);
                        ss = fmaf(o, o, ss);
                    }
                }
            }
            ctl->ss_part[m][row] = ss;
            named_bar_sync(pair_bar, 64);
            float ss_tot = ctl->ss_part[0][row] + ctl->ss_part[1][row];
            if (p.nslices == 2) {
                const int pb = r & 1;
                if (m == 0) {
                    st_cluster_f32(&ctl->ss_peer[pb][row], cluster_ctarank() ^ 1u, ss_tot);
                    mbar_arrive_remote(&ctl->peer_bar[pb], cluster_ctarank() ^ 1u);
                }
                if (!mbar_wait_cluster(&ctl->peer_bar[pb], (r >> 1) & 1, p.err, abort_flag)) ok = false;
                ss_tot += ctl->ss_peer[pb][row];
            }
            ok = __all_sync(0xffffffffu, ok);
            const float yscale =
                p.no_norm ? 1.f : (1.f - p.lambda_init) * rsqrtf(ss_tot / static_cast<float>(p.dv) + p.eps);
            if (ok) {
                if constexpr (LY::TMA_OUT) {
                    // stage this warp's 32 rows x 64 columns (128-byte swizzle:
                    // 16-byte chunk c of row t sits at chunk c ^ (t % 8)) and
                    // write them with one TMA store; rows past L are clipped
                    uint8_t *obuf = smem + LY::OFF_OUT + (warp - 2) * (32 * 128);
                    if (lane == 0) bulk_wait_group_read0();   // the previous item's store has read it
                    __syncwarp();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t r1[32], r2[32];
                        tmem_ld32(tO1 + col0 + cc * 32, r1);
                        tmem_ld32(tO2 + col0 + cc * 32, r2);
                        tmem_ld_wait_regs(r1);
                        reg_fence(r2);
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float y0 = (__fmul_rn(__uint_as_float(r1[e]), inv1) -
                                              __fmul_rn(__uint_as_float(r2[e]), c2)) * yscale;
                            const float y1 = (__fmul_rn(__uint_as_float(r1[e + 1]), inv1) -
                                              __fmul_rn(__uint_as_float(r2[e + 1]), c2)) * yscale;
                            pk[e / 2] = pack_bf16x2(y0, y1);
                        }
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            const int ch = cc * 4 + v4;
                            *reinterpret_cast<uint4 *>(obuf + lane * 128 + ((ch ^ (lane & 7)) * 16)) =
                                make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_4d(&tmO, obuf, slice * kDVS + col0, it.h, it.q0 + quarter * 32, it.b);
                        bulk_commit_group();
                    }
                } else {
                    __nv_bfloat16 *orow =
                        p.out + ((static_cast<size_t>(it.b) * p.L + qrow) * p.hs + it.h) * p.dv + slice * kDVS + col0;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t r1[32], r2[32];
                        tmem_ld32(tO1 + col0 + cc * 32, r1);
                        tmem_ld32(tO2 + col0 + cc * 32, r2);
                        tmem_ld_wait_regs(r1);
                        reg_fence(r2);
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float y0 = (__fmul_rn(__uint_as_float(r1[e]), inv1) -
                                              __fmul_rn(__uint_as_float(r2[e]), c2)) * yscale;
                            const float y1 = (__fmul_rn(__uint_as_float(r1[e + 1]), inv1) -
                                              __fmul_rn(__uint_as_float(r2[e + 1]), c2)) * yscale;
                            pk[e / 2] = pack_bf16x2(y0, y1);
                        }
                        if (qrow < p.L) {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4)
                                dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                        }
                    }
                }
            }
            // the accumulators may now be overwritten by the next item's first PV
            tc_fence_before();
            mbar_arrive(&ctl->o_free);
            gt += nkv;
            // both warps of the pair agree on whether to go on; pairs share no
            // named barrier, so one that stops early cannot block another
            // (every mbarrier wait is bounded and sees the abort flag)
            if (bar_red_or(pair_bar, 64, !ok || *abort_flag)) break;
        }
    }

    // ---- teardown: our TMA stores have read their staging buffers, and all
    // TMEM traffic of this CTA is complete past this barrier
    if (LY::TMA_OUT && warp >= 2 && lane == 0) bulk_wait_group0();
    tc_fence_before();
    __syncthreads();
    if (p.nslices == 2) cluster_sync_all();   // no DSMEM traffic into an exited peer
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
int launch_impl(const PrefillArgs &a, cudaStream_t stream) {
    using LY = Layout<D>;
    CUtensorMap mQ1, mK1, mQ2, mK2, mV, mO;
    // queries and output: L rows; keys and values: Lk rows
    const uint64_t B = a.B, L = a.L, Lk = a.Lk > 0 ? a.Lk : a.L, hs = a.hs, hn = a.hn, d = a.d, dv = a.dv;
    {
        const uint64_t dq[4] = {d, hs, L, B}, dk[4] = {d, hs, Lk, B};
        const uint64_t sq[3] = {d * 2, hs * d * 2, L * hs * d * 2}, sk[3] = {d * 2, hs * d * 2, Lk * hs * d * 2};
        const uint32_t boxq[4] = {64, 1, kBM, 1};
        const uint32_t boxk[4] = {64, 1, (uint32_t)LY::BN, 1};
        if (!encode_tmap_4d_bf16(&mQ1, a.q1, dq, sq, boxq)) return GDA_ERR_CUDA;
        if (!encode_tmap_4d_bf16(&mK1, a.k1, dk, sk, boxk)) return GDA_ERR_CUDA;
    }
    {
        const uint64_t dq[4] = {d, hn, L, B}, dk[4] = {d, hn, Lk, B};
        const uint64_t sq[3] = {d * 2, hn * d * 2, L * hn * d * 2}, sk[3] = {d * 2, hn * d * 2, Lk * hn * d * 2};
        const uint32_t boxq[4] = {64, 1, kBM, 1};
        const uint32_t boxk[4] = {64, 1, (uint32_t)LY::BN, 1};
        if (!encode_tmap_4d_bf16(&mQ2, a.q2, dq, sq, boxq)) return GDA_ERR_CUDA;
        if (!encode_tmap_4d_bf16(&mK2, a.k2, dk, sk, boxk)) return GDA_ERR_CUDA;
    }
    {
        const uint64_t dk[4] = {dv, hs, Lk, B};
        const uint64_t sk[3] = {dv * 2, hs * dv * 2, Lk * hs * dv * 2};
        const uint32_t box[4] = {64, 1, (uint32_t)LY::BN, 1};
        if (!encode_tmap_4d_bf16(&mV, a.v, dk, sk, box)) return GDA_ERR_CUDA;
        // output: 32 query rows x 64 columns of one head per store
        const uint64_t dq[4] = {dv, hs, L, B};
        const uint64_t sq[3] = {dv * 2, hs * dv * 2, L * hs * dv * 2};
        const uint32_t boxo[4] = {64, 1, 32, 1};
        if (!encode_tmap_4d_bf16(&mO, a.out, dq, sq, boxo)) return GDA_ERR_CUDA;
    }
    TcParams p;
    p.lambda = a.lambda;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.err = a.dev_err;
    p.lambda_init = a.lambda_init;
    p.eps = a.eps;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.d)));
    p.B = a.B;
    p.L = a.L;
    p.Lk = static_cast<int>(Lk);
    p.koff = static_cast<int>(Lk) - a.L;
    p.hs = a.hs;
    p.hn = a.hn;
    p.dv = a.dv;
    p.causal = a.causal;
    p.nslices = a.dv / kDVS;
    p.nqt = (a.L + kBM - 1) / kBM;
    p.no_norm = (a.flags & GDA_FLAG_NO_NORM) ? 1 : 0;

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    auto kern = gda_prefill_tc_kernel<D>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::TOTAL);
    if (e != cudaSuccess) return record_cuda_error(e);
    const long long nitems = static_cast<long long>(p.nqt) * a.B * a.hs;
    if (nitems <= 0 || nitems > 0x7fffffffLL) return GDA_ERR_UNSUPPORTED;
    // one CTA (or CTA pair) per SM (pair of SMs), never more than there are items
    long long groups = sms / p.nslices;
    if (groups < 1) groups = 1;
    if (groups > nitems) groups = nitems;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(groups * p.nslices), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = LY::TOTAL;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.nslices;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mQ1, mK1, mQ2, mK2, mV, mO, p);
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

}  // namespace

int launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream) {
    if (a.d == 64) return launch_impl<64>(a, stream);
    if (a.d == 128) return launch_impl<128>(a, stream);
    return GDA_ERR_UNSUPPORTED;
}

}  // namespace gda
