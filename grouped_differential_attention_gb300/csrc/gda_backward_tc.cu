// Gradients of grouped differential attention on the tensor cores (bf16
// operands, float32 accumulation in TMEM), d = 64, dv = 128.
//
// Forward (per batch b, signal head h, noise head g = h / r, query row i;
// "Differential Attention in Large Language Models ...", sections
// "Differential Attention Architecture" and "Headwise Normalization"; noise
// heads shared by groups per the "Grouped Differential Attention" abstract):
//   a1 = softmax_j(q1_i . k1_j / sqrt d),  a2 = softmax_j(q2_i . k2_j / sqrt d)
//   O1 = sum_j a1_j v_j,  O2 = sum_j a2_j v_j,  o = O1 - lambda_h O2
//   y = (1 - lambda_init) o / rms,  rms = sqrt(mean(o^2) + eps)
// Backward of sum(dy . y):
//   do = (c / rms)(dy - o (dy . o) / (dv rms^2))    (c = 1 - lambda_init; do = dy without the norm)
//   dP_ij = do_i . v_j,  D1_i = do_i . O1_i,  D2_i = do_i . O2_i
//   dS1 = a1 (dP - D1),  dS2 = -lambda_h a2 (dP - D2),  W = a1 - lambda_h a2
//   dv_j = sum_i W_ij do_i;  dk1_j = sum_i dS1_ij q1_i / sqrt d;  dq1_i = sum_j dS1_ij k1_j / sqrt d
//   dk2, dq2: the same with dS2, q2, k2, summed over the r signal heads of the group
//   dlambda_h = -sum_{b,i} D2_i
//
// Kernels (all persistent, roles as in the prefill kernels: warp 0 TMA
// producer, warp 1 TMEM allocator + single-thread MMA issuer, warps 2-17 the
// elementwise threads, warps 2 + 4c .. 5 + 4c taking the 16-column group c of
// each 64-column tile):
//   pass 1 (gda_lse_tc_kernel, shared with the two-pass prefill): base-2
//          log-sum-exp of every signal and noise map row;
//   prep   (gda_bwd_prep_kernel): per (128 query rows, b, h) both maps with
//          their final statistics, O1 and O2 in two TMEM accumulators; the
//          epilogue forms o, the norm's input gradient do (rounded to bf16,
//          written for the later MMAs), D1 and D2 from the rounded do;
//   dK/dV  (gda_bwd_dkdv_kernel): per (128 keys, b, noise group), thread =
//          key: S1^T, S2^T and dP^T = V dO^T on the tensor core, W / dS1 /
//          dS2 in registers from the saved statistics, then dV += W dO,
//          dK1 += dS1 Q1, dK2 += dS2 Q2 with the A operand in TMEM; dK2
//          accumulates over the group's heads in TMEM (no atomics);
//   dQ     (gda_bwd_dq_kernel): per (128 query rows, b, noise group), thread
//          = query row: S1, S2, dP = dO V^T, then dQ1 += dS1 K1 and
//          dQ2 += dS2 K2 (dQ2 accumulated over the group's heads);
//   reduce (gda_bwd_dlambda_kernel): dlambda in a fixed order.
// Every mbarrier wait is bounded (1 s, GDA_DEVERR_PREFILL_TIMEOUT).
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

constexpr int kD = 64;
constexpr int kDV = 128;
constexpr int kN = 64;             // N-side tile

struct BwdTcParams {
    const float *lambda;
    const float *lse;              // [B, hs + hn, Lp] base-2 log-sum-exp
    const __nv_bfloat16 *dy;       // [B, L, hs, dv]
    __nv_bfloat16 *dO;             // [B, L, hs, dv]
    float *D1, *D2;                // [B, hs, Lp]
    float *dq1, *dk1, *dq2, *dk2, *dvo, *dlambda;
    unsigned *err;
    float lambda_init, eps, scale_log2, scale;
    int B, L, Lp, hs, hn, causal, no_norm;
};

__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// TS MMA: D[128 x N] (+)= A[128 x 64] B[64 x N]; A = bf16 pairs in TMEM,
// written by four 16-column groups (K rows 16k .. 16k+15 in TMEM columns
// tA + 16k .. tA + 16k + 7); B = MN-major smem tile of 64 K-rows, N/64
// column blocks 8 KiB apart (128-byte rows, 128-byte swizzle).
template <int N>
__device__ __forceinline__ void issue_ts64q(uint32_t tD, uint32_t tA, uint32_t ba, bool acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, N, 1);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint64_t b = smem_desc_sw128(ba + k * 2048, 64 * 128, 1024);
        mma_ts(tD, tA + k * 16, b, idesc, (acc || k > 0) ? 1u : 0u);
    }
}

// D[128 x N] (+)= A[128 x 64] B[64 x N]: A a K-major shared-memory tile
// (128-byte rows, 128-byte swizzle), B as in issue_ts64.
template <int N>
__device__ __forceinline__ void issue_ss64(uint32_t tD, uint32_t aa, uint32_t ba, bool acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, N, 1);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint64_t a = smem_desc_sw128(aa + k * 32, 16, 1024);
        const uint64_t b = smem_desc_sw128(ba + k * 2048, 64 * 128, 1024);
        mma_ss(tD, a, b, idesc, (acc || k > 0) ? 1u : 0u);
    }
}

// S[128 x 64] = A[128 x K] B[64 x K]^T with K-major operands: A in K/64
// blocks of [128 x 64] (16 KiB apart), B in K/64 blocks of [64 x 64] (8 KiB apart).
template <int K>
__device__ __forceinline__ void issue_nt(uint32_t tS, uint32_t aa, uint32_t ba) {
    issue_qk<K, kN>(tS, aa, ba);
}

// 32 lanes x 32 bit, 8 consecutive columns per thread.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// ================================================================ prep ==

struct PrepLayout {
    static constexpr int KS = 4, VS = 4;
    static constexpr int Q_BYTES = kBM * kD * 2;          // 16 KiB
    static constexpr int K_BYTES = kN * kD * 2;           // 8 KiB
    static constexpr int KST_BYTES = 2 * K_BYTES;
    static constexpr int V_BYTES = kN * kDV * 2;          // 16 KiB
    static constexpr int OFF_Q1 = 0, OFF_Q2 = Q_BYTES, OFF_K = 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KS * KST_BYTES;
    static constexpr int TILES = OFF_V + VS * V_BYTES;
};

struct PrepCtrl {
    uint64_t q_full, q_empty;
    uint64_t k_full[4], k_empty[4];
    uint64_t v_full[4], v_empty[4];
    uint64_t s_full[2], p_full[2];
    uint64_t o_final, o_free, mma_idle;
    uint32_t tmem_base;
    int abort_flag;
    float x1[4][kBM], x2[4][kBM];      // per-group partial sums, exchange 1 (ss, dy.o)
    float y1[4][kBM], y2[4][kBM];      // exchange 2 (D1, D2)
};

constexpr int prep_smem_bytes() {
    return PrepLayout::TILES + static_cast<int>((sizeof(PrepCtrl) + 1023) / 1024) * 1024 + 1024;
}

// (query tile, b, h) items, last query tiles first
__device__ __forceinline__ bool prep_item(const BwdTcParams &p, int r, int G, int cid, int &b, int &h, int &q0,
                                          int &nkv) {
    const int nqt = (p.L + kBM - 1) / kBM;
    const int per = p.B * p.hs;
    const long long n = static_cast<long long>(nqt) * per;
    const int k = (r & 1) ? (G - 1 - cid) : cid;
    const long long idx = static_cast<long long>(r) * G + k;
    if (idx >= n) return false;
    const int i = static_cast<int>(idx);
    q0 = (nqt - 1 - i / per) * kBM;
    b = (i % per) / p.hs;
    h = (i % per) % p.hs;
    const int kv_end = p.causal ? min(p.L, q0 + kBM) : p.L;
    nkv = (kv_end + kN - 1) / kN;
    return true;
}

// Bounded wait that first polls without the suspend-time hint (a wait whose phase has
// already completed costs about a third as much that way, which matters on the
// single-thread MMA issuers), then falls back to the bounded hinted wait.
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

// Kernels after the first are programmatic dependent launches: each sets up its barriers
// and TMEM while the previous kernel finishes, then waits here for that grid's completion
// (its writes visible) before reading anything it produced.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                             cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr int kEwP = 512;           // prep elementwise threads: 16 warps, four column groups
constexpr int kThrP = 64 + kEwP;

__global__ void __launch_bounds__(kThrP, 1)
gda_bwd_prep_kernel(const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmK1,
                    const __grid_constant__ CUtensorMap tmQ2, const __grid_constant__ CUtensorMap tmK2,
                    const __grid_constant__ CUtensorMap tmV, const BwdTcParams p) {
    using LY = PrepLayout;
    constexpr int KS = LY::KS, VS = LY::VS;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, offset from the shared array itself so that accesses stay in the
    // shared state space (32-bit addresses)
    uint8_t *smem = smem_raw + ((0u - smem_u32(smem_raw)) & 1023u);
    PrepCtrl *ctl = reinterpret_cast<PrepCtrl *>(smem + LY::TILES);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cid = blockIdx.x, G = gridDim.x;
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
            mbar_init(&ctl->p_full[bb], kEwP);
        }
        mbar_init(&ctl->o_final, 1);
        mbar_init(&ctl->o_free, kEwP);
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
    griddep_wait();      // the previous kernel's outputs (launched as its programmatic dependent)
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;
    // TMEM: O1 [0,128) | O2 [128,256) | S1 x 2 [256,384) | S2 x 2 [384,512)
    constexpr uint32_t tO2 = 128, tS1_0 = 256, tS2_0 = 384;

    if (warp == 0) {
        if (elect_one()) {
            tma_prefetch_desc(&tmQ1);
            tma_prefetch_desc(&tmK1);
            tma_prefetch_desc(&tmQ2);
            tma_prefetch_desc(&tmK2);
            tma_prefetch_desc(&tmV);
            uint32_t kt = 0, vt = 0;
            int nq = 0;
            bool ok = true;
            int b, h, q0, nkv;
            for (int r = 0; ok && prep_item(p, r, G, cid, b, h, q0, nkv); ++r) {
                const int g = h / r_grp;
                if (r > 0 && !wait_quick(&ctl->q_empty, (r - 1) & 1, p.err, abort_flag)) break;
                mbar_arrive_expect_tx(&ctl->q_full, 2 * LY::Q_BYTES);
                tma_load_4d(smem + LY::OFF_Q1, &tmQ1, &ctl->q_full, 0, h, q0, b);
                tma_load_4d(smem + LY::OFF_Q2, &tmQ2, &ctl->q_full, 0, g, q0, b);
                ++nq;
                auto load_k = [&](int j) -> bool {
                    const uint32_t gk = kt + j;
                    const int st = gk % KS;
                    if (gk >= KS && !wait_quick(&ctl->k_empty[st], ((gk / KS) - 1) & 1, p.err, abort_flag))
                        return false;
                    uint8_t *sb = smem + LY::OFF_K + st * LY::KST_BYTES;
                    mbar_arrive_expect_tx(&ctl->k_full[st], LY::KST_BYTES);
                    tma_load_4d(sb, &tmK1, &ctl->k_full[st], 0, h, j * kN, b);
                    tma_load_4d(sb + LY::K_BYTES, &tmK2, &ctl->k_full[st], 0, g, j * kN, b);
                    return true;
                };
                auto load_v = [&](int j) -> bool {
                    const uint32_t gv = vt + j;
                    const int st = gv % VS;
                    if (gv >= VS && !wait_quick(&ctl->v_empty[st], ((gv / VS) - 1) & 1, p.err, abort_flag))
                        return false;
                    uint8_t *sb = smem + LY::OFF_V + st * LY::V_BYTES;
                    mbar_arrive_expect_tx(&ctl->v_full[st], LY::V_BYTES);
                    tma_load_4d(sb, &tmV, &ctl->v_full[st], 0, h, j * kN, b);
                    tma_load_4d(sb + kN * 128, &tmV, &ctl->v_full[st], 64, h, j * kN, b);
                    return true;
                };
                int kdone = 0, vdone = 0;
                for (int t = 0; ok && t < 2 && t < nkv; ++t) {
                    ok = load_k(t);
                    if (ok) ++kdone;
                }
                for (int j = 0; ok && j < nkv; ++j) {
                    if (j + 2 < nkv) {
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
        if (elect_one()) {
            const uint32_t q1a = smem_u32(smem + LY::OFF_Q1), q2a = smem_u32(smem + LY::OFF_Q2);
            const uint32_t k0a = smem_u32(smem + LY::OFF_K), v0a = smem_u32(smem + LY::OFF_V);
            uint32_t kt = 0, vt = 0, gt = 0;
            bool ok = true;
            int b, h, q0, nkv;
            for (int r = 0; ok && prep_item(p, r, G, cid, b, h, q0, nkv); ++r) {
                if (!wait_quick(&ctl->q_full, r & 1, p.err, abort_flag)) break;
                for (int t = 0; t < 2 && t < nkv; ++t) {
                    const uint32_t gk = kt + t, gs = gt + t;
                    if (!wait_quick(&ctl->k_full[gk % KS], (gk / KS) & 1, p.err, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ka = k0a + (gk % KS) * LY::KST_BYTES;
                    issue_qk<kD, kN>(tmem + tS1_0 + (gs & 1) * kN, q1a, ka);
                    issue_qk<kD, kN>(tmem + tS2_0 + (gs & 1) * kN, q2a, ka + LY::K_BYTES);
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
                    const uint32_t va = v0a + (gv % VS) * LY::V_BYTES;
                    issue_ts64q<kDV>(tmem, tmem + tS1_0 + bb * kN, va, j > 0);
                    issue_ts64q<kDV>(tmem + tO2, tmem + tS2_0 + bb * kN, va, j > 0);
                    mma_commit(&ctl->v_empty[gv % VS]);
                    const int jn = j + 2;
                    if (jn < nkv) {
                        const uint32_t gk = kt + jn;
                        if (!wait_quick(&ctl->k_full[gk % KS], (gk / KS) & 1, p.err, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t ka = k0a + (gk % KS) * LY::KST_BYTES;
                        issue_qk<kD, kN>(tmem + tS1_0 + bb * kN, q1a, ka);
                        issue_qk<kD, kN>(tmem + tS2_0 + bb * kN, q2a, ka + LY::K_BYTES);
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
        const int grp = (warp - 2) / 4;             // key columns [16 grp, +16) of each tile; dv columns [32 grp, +32)
        const int quarter = warp % 4;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        const int heads = p.hs + p.hn;
        uint32_t gt = 0;
        int b, h, q0, nkv;
        for (int r = 0; prep_item(p, r, G, cid, b, h, q0, nkv); ++r) {
            const int g = h / r_grp;
            const int qrow = q0 + row;
            const bool in = qrow < p.L;
            const int last_key = p.causal ? min(qrow, p.L - 1) : p.L - 1;
            const float lam = p.lambda[h];
            const float neg1 = in ? -p.lse[(static_cast<size_t>(b) * heads + h) * p.Lp + qrow] : -INFINITY;
            const float neg2 = in ? -p.lse[(static_cast<size_t>(b) * heads + p.hs + g) * p.Lp + qrow] : -INFINITY;
            // this thread's 32 dy values, requested now so the loads complete during the tile loop
            const int c0 = grp * 32;
            const size_t rowix = (static_cast<size_t>(b) * p.L + (in ? qrow : 0)) * p.hs + h;
            uint4 dyv[4];
            {
                const uint4 *dyrow = reinterpret_cast<const uint4 *>(p.dy + rowix * kDV + c0);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) dyv[v4] = in ? dyrow[v4] : make_uint4(0, 0, 0, 0);
            }
            bool ok = true;
            for (int j = 0; j < nkv; ++j) {
                const uint32_t gs = gt + j;
                const int bb = gs & 1;
                // per-lane waits: a failed one sets the error word and the flag that ends every
                // later wait at once; the loop runs on, so the barrier counts stay whole
                if (!wait_quick(&ctl->s_full[bb], (gs >> 1) & 1, p.err, abort_flag)) ok = false;
                tc_fence_after();
                const uint32_t tS1 = tmem + lane_off + tS1_0 + bb * kN + grp * 16;
                const uint32_t tS2 = tmem + lane_off + tS2_0 + bb * kN + grp * 16;
                uint32_t r1[16], r2[16];
                tmem_ld16(tS1, r1);
                tmem_ld16(tS2, r2);
                tmem_ld_wait_regs16(r1);
                reg_fence16(r2);
                const int k0 = j * kN + grp * 16;
                uint32_t pk1[8], pk2[8];
                auto probs = [&](auto masked) {
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        float x0 = __uint_as_float(r1[e]), x1 = __uint_as_float(r1[e + 1]);
                        float y0 = __uint_as_float(r2[e]), y1 = __uint_as_float(r2[e + 1]);
                        ffma2(x0, x1, sl2, sl2, neg1, neg1);
                        ffma2(y0, y1, sl2, sl2, neg2, neg2);
                        x0 = fast_exp2(x0);
                        x1 = fast_exp2(x1);
                        y0 = fast_exp2(y0);
                        y1 = fast_exp2(y1);
                        if constexpr (decltype(masked)::value) {
                            if (k0 + e > last_key) x0 = y0 = 0.f;
                            if (k0 + e + 1 > last_key) x1 = y1 = 0.f;
                        }
                        pk1[e / 2] = pack_bf16x2(x0, x1);
                        pk2[e / 2] = pack_bf16x2(y0, y1);
                    }
                };
                // the per-key test only where some row of the warp has keys past its last one
                if (__any_sync(0xffffffffu, k0 + 15 > last_key))
                    probs(std::true_type{});
                else
                    probs(std::false_type{});
                tmem_st8(tS1, pk1);
                tmem_st8(tS2, pk2);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&ctl->p_full[bb]);
            }
            tmem_ld_wait();

            // ---- epilogue: o, the norm's input gradient, D1, D2 (this group: 32 dv columns)
            ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
            if (ok) ok = warp_wait(&ctl->o_final, r & 1, p.err, abort_flag);
            tc_fence_after();
            float ss = 0.f, dyo = 0.f;
            if (ok) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t o1[16], o2[16];
                    tmem_ld16(tmem + lane_off + c0 + cc * 16, o1);
                    tmem_ld16(tmem + lane_off + tO2 + c0 + cc * 16, o2);
                    tmem_ld_wait_regs16(o1);
                    reg_fence16(o2);
                    const uint32_t *dw = reinterpret_cast<const uint32_t *>(&dyv[cc * 2]);
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const float oa = __uint_as_float(o1[e]) - __fmul_rn(__uint_as_float(o2[e]), lam);
                        const float ob = __uint_as_float(o1[e + 1]) - __fmul_rn(__uint_as_float(o2[e + 1]), lam);
                        ss = fmaf(oa, oa, fmaf(ob, ob, ss));
                        dyo = fmaf(bf_lo(dw[e / 2]), oa, fmaf(bf_hi(dw[e / 2]), ob, dyo));
                    }
                }
            }
            ctl->x1[grp][row] = ss;
            ctl->x2[grp][row] = dyo;
            named_bar_sync(1, kEwP);
            ok = __all_sync(0xffffffffu, ok);
            const float ss_t = (ctl->x1[0][row] + ctl->x1[1][row]) + (ctl->x1[2][row] + ctl->x1[3][row]);
            const float dyo_t = (ctl->x2[0][row] + ctl->x2[1][row]) + (ctl->x2[2][row] + ctl->x2[3][row]);
            float a = 1.f, bc = 0.f;                    // do = a dy - bc o
            if (!p.no_norm) {
                const float r2 = ss_t / static_cast<float>(kDV) + p.eps;
                a = (1.f - p.lambda_init) * rsqrtf(r2);
                bc = a * dyo_t / (static_cast<float>(kDV) * r2);
            }
            float d1 = 0.f, d2 = 0.f;
            if (ok) {
                uint4 *dorow = reinterpret_cast<uint4 *>(p.dO + rowix * kDV + c0);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t o1[16], o2[16];
                    tmem_ld16(tmem + lane_off + c0 + cc * 16, o1);
                    tmem_ld16(tmem + lane_off + tO2 + c0 + cc * 16, o2);
                    tmem_ld_wait_regs16(o1);
                    reg_fence16(o2);
                    const uint32_t *dw = reinterpret_cast<const uint32_t *>(&dyv[cc * 2]);
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const float O1a = __uint_as_float(o1[e]), O1b = __uint_as_float(o1[e + 1]);
                        const float O2a = __uint_as_float(o2[e]), O2b = __uint_as_float(o2[e + 1]);
                        const float oa = O1a - __fmul_rn(O2a, lam);
                        const float ob = O1b - __fmul_rn(O2b, lam);
                        const uint32_t w = pack_bf16x2(a * bf_lo(dw[e / 2]) - bc * oa, a * bf_hi(dw[e / 2]) - bc * ob);
                        pk[e / 2] = w;
                        // D from the rounded do, the value the later products use
                        d1 = fmaf(bf_lo(w), O1a, fmaf(bf_hi(w), O1b, d1));
                        d2 = fmaf(bf_lo(w), O2a, fmaf(bf_hi(w), O2b, d2));
                    }
                    if (in) {
#pragma unroll
                        for (int v4 = 0; v4 < 2; ++v4)
                            dorow[cc * 2 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    }
                }
            }
            ctl->y1[grp][row] = d1;
            ctl->y2[grp][row] = d2;
            named_bar_sync(1, kEwP);
            if (grp == 0 && in && ok) {
                const size_t vix = (static_cast<size_t>(b) * p.hs + h) * p.Lp + qrow;
                p.D1[vix] = (ctl->y1[0][row] + ctl->y1[1][row]) + (ctl->y1[2][row] + ctl->y1[3][row]);
                p.D2[vix] = (ctl->y2[0][row] + ctl->y2[1][row]) + (ctl->y2[2][row] + ctl->y2[3][row]);
            }
            tc_fence_before();
            mbar_arrive(&ctl->o_free);
            gt += nkv;
            if (bar_red_or(1, kEwP, !ok || *abort_flag)) break;
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

// =============================================================== dK / dV ==
// Item = (128-key tile, b, noise group g); inside: the group's r signal heads,
// each over the 64-row query tiles that see the keys.

struct KvLayout {
    static constexpr int QS = 3;
    static constexpr int K_BYTES = kBM * kD * 2;          // K1_h or K2_g tile: 16 KiB
    static constexpr int V_BYTES = kBM * kDV * 2;         // 32 KiB (two [128 x 64] blocks)
    static constexpr int Q_BYTES = kN * kD * 2;           // Q1 / Q2 tile: 8 KiB
    static constexpr int DO_BYTES = kN * kDV * 2;         // 16 KiB (two [64 x 64] blocks)
    static constexpr int VEC_BYTES = 4 * kN * 4;          // lse1, lse2, D1, D2 of 64 rows
    static constexpr int QST_BYTES = 2 * Q_BYTES + DO_BYTES + 1024;   // vectors padded to 1 KiB
    static constexpr int OFF_K1 = 0, OFF_K2 = K_BYTES, OFF_V = 2 * K_BYTES;
    static constexpr int OFF_Q = OFF_V + V_BYTES;
    static constexpr int W_BYTES = kBM * kN * 2;          // one of W / dS1 / dS2: 16 KiB
    static constexpr int OFF_W = OFF_Q + QS * QST_BYTES;  // W | dS1 | dS2, K-major, 128-byte swizzle
    static constexpr int TILES = OFF_W + 3 * W_BYTES;
};

struct KvCtrl {
    uint64_t g_full, g_empty;        // K2 of the item
    uint64_t h_full, h_empty;        // K1 and V of the current head
    uint64_t q_full[3], q_empty[3];  // query-side stages
    uint64_t s_full, s_free;         // S^T tiles in TMEM / read into registers
    uint64_t p_full, w_free;         // W, dS1, dS2 in shared memory / read by their products
    uint64_t acc_ready, acc_free;    // dV, dK1 of a head
    uint64_t k2_ready, k2_free;      // dK2 of an item
    uint64_t mma_idle;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr int kv_smem_bytes() {
    return KvLayout::TILES + static_cast<int>((sizeof(KvCtrl) + 1023) / 1024) * 1024 + 1024;
}

// (key tile, b, g) items, first key tiles (most query rows) first
__device__ __forceinline__ bool kv_item(const BwdTcParams &p, int r, int G, int cid, int &b, int &g, int &k0,
                                        int &i0, int &nq) {
    const int nkt = (p.L + kBM - 1) / kBM;
    const int per = p.B * p.hn;
    const long long n = static_cast<long long>(nkt) * per;
    const int k = (r & 1) ? (G - 1 - cid) : cid;
    const long long idx = static_cast<long long>(r) * G + k;
    if (idx >= n) return false;
    const int i = static_cast<int>(idx);
    k0 = (i / per) * kBM;
    b = (i % per) / p.hn;
    g = (i % per) % p.hn;
    const int nq64 = (p.L + kN - 1) / kN;
    i0 = p.causal ? k0 / kN : 0;
    nq = nq64 - i0;
    return true;
}

constexpr int kEwKv = 512;          // dK/dV elementwise threads: 16 warps, four 16-column groups
constexpr int kThrKv = 64 + kEwKv;

__global__ void __launch_bounds__(kThrKv, 1)
gda_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmK1, const __grid_constant__ CUtensorMap tmK2,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQ1,
                    const __grid_constant__ CUtensorMap tmQ2, const __grid_constant__ CUtensorMap tmdO,
                    const BwdTcParams p) {
    using LY = KvLayout;
    constexpr int QS = LY::QS;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, offset from the shared array itself so that accesses stay in the
    // shared state space (32-bit addresses)
    uint8_t *smem = smem_raw + ((0u - smem_u32(smem_raw)) & 1023u);
    KvCtrl *ctl = reinterpret_cast<KvCtrl *>(smem + LY::TILES);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cid = blockIdx.x, G = gridDim.x;
    const int r_grp = p.hs / p.hn;
    const int heads = p.hs + p.hn;

    if (threadIdx.x == 0) {
        mbar_init(&ctl->g_full, 1);
        mbar_init(&ctl->g_empty, 1);
        mbar_init(&ctl->h_full, 1);
        mbar_init(&ctl->h_empty, 1);
        for (int s = 0; s < QS; ++s) {
            mbar_init(&ctl->q_full[s], 1);
            mbar_init(&ctl->q_empty[s], 1);
        }
        mbar_init(&ctl->s_full, 1);
        mbar_init(&ctl->s_free, kEwKv);
        mbar_init(&ctl->p_full, kEwKv);
        mbar_init(&ctl->w_free, 1);
        mbar_init(&ctl->acc_ready, 1);
        mbar_init(&ctl->acc_free, kEwKv);
        mbar_init(&ctl->k2_ready, 1);
        mbar_init(&ctl->k2_free, kEwKv);
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
    griddep_wait();      // the previous kernel's outputs (launched as its programmatic dependent)
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;
    // TMEM: S1^T [0,64) | S2^T [64,128) | dP^T [128,192) | dV [192,320) | dK1 [320,384) | dK2 [384,448)
    constexpr uint32_t tS1 = 0, tS2 = 64, tdP = 128, tdV = 192, tdK1 = 320, tdK2 = 384;

    if (warp == 0) {
        if (elect_one()) {
            tma_prefetch_desc(&tmK1);
            tma_prefetch_desc(&tmK2);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmQ1);
            tma_prefetch_desc(&tmQ2);
            tma_prefetch_desc(&tmdO);
            uint32_t gq = 0, nh = 0;
            int ng = 0;
            bool ok = true;
            int b, g, k0, i0, nq;
            for (int r = 0; ok && kv_item(p, r, G, cid, b, g, k0, i0, nq); ++r) {
                if (r > 0 && !wait_quick(&ctl->g_empty, (r - 1) & 1, p.err, abort_flag)) break;
                mbar_arrive_expect_tx(&ctl->g_full, LY::K_BYTES);
                tma_load_4d(smem + LY::OFF_K2, &tmK2, &ctl->g_full, 0, g, k0, b);
                ++ng;
                for (int hi = 0; ok && hi < r_grp; ++hi) {
                    const int h = g * r_grp + hi;
                    if (nh > 0 && !wait_quick(&ctl->h_empty, (nh - 1) & 1, p.err, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&ctl->h_full, LY::K_BYTES + LY::V_BYTES);
                    tma_load_4d(smem + LY::OFF_K1, &tmK1, &ctl->h_full, 0, h, k0, b);
                    tma_load_4d(smem + LY::OFF_V, &tmV, &ctl->h_full, 0, h, k0, b);
                    tma_load_4d(smem + LY::OFF_V + kBM * 128, &tmV, &ctl->h_full, 64, h, k0, b);
                    ++nh;
                    for (int i = 0; i < nq; ++i) {
                        const int q0 = (i0 + i) * kN;
                        const int st = gq % QS;
                        if (gq >= QS && !wait_quick(&ctl->q_empty[st], ((gq / QS) - 1) & 1, p.err, abort_flag)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sb = smem + LY::OFF_Q + st * LY::QST_BYTES;
                        mbar_arrive_expect_tx(&ctl->q_full[st], 2 * LY::Q_BYTES + LY::DO_BYTES + LY::VEC_BYTES);
                        tma_load_4d(sb, &tmQ1, &ctl->q_full[st], 0, h, q0, b);
                        tma_load_4d(sb + LY::Q_BYTES, &tmQ2, &ctl->q_full[st], 0, g, q0, b);
                        tma_load_4d(sb + 2 * LY::Q_BYTES, &tmdO, &ctl->q_full[st], 0, h, q0, b);
                        tma_load_4d(sb + 2 * LY::Q_BYTES + kN * 128, &tmdO, &ctl->q_full[st], 64, h, q0, b);
                        float *vec = reinterpret_cast<float *>(sb + 2 * LY::Q_BYTES + LY::DO_BYTES);
                        bulk_g2s(vec, p.lse + (static_cast<size_t>(b) * heads + h) * p.Lp + q0, 256, &ctl->q_full[st]);
                        bulk_g2s(vec + 64, p.lse + (static_cast<size_t>(b) * heads + p.hs + g) * p.Lp + q0, 256,
                                 &ctl->q_full[st]);
                        bulk_g2s(vec + 128, p.D1 + (static_cast<size_t>(b) * p.hs + h) * p.Lp + q0, 256, &ctl->q_full[st]);
                        bulk_g2s(vec + 192, p.D2 + (static_cast<size_t>(b) * p.hs + h) * p.Lp + q0, 256, &ctl->q_full[st]);
                        ++gq;
                    }
                }
            }
            if (ng > 0) drain_wait(&ctl->g_full, (ng - 1) & 1, p.err);
            if (nh > 0) drain_wait(&ctl->h_full, (nh - 1) & 1, p.err);
            for (uint32_t j = (gq > QS ? gq - QS : 0); j < gq; ++j)
                drain_wait(&ctl->q_full[j % QS], (j / QS) & 1, p.err);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (elect_one()) {
            const uint32_t k1a = smem_u32(smem + LY::OFF_K1), k2a = smem_u32(smem + LY::OFF_K2);
            const uint32_t va = smem_u32(smem + LY::OFF_V), q0a = smem_u32(smem + LY::OFF_Q);
            const uint32_t wa = smem_u32(smem + LY::OFF_W);
            uint32_t gq = 0, nh = 0;
            bool ok = true;
            int b, g, k0, i0, nq;
            // dV, dK1 and dK2 updates of tile t (tile i of head hi of item r); they run
            // after the logits of tile t + 1 were issued, so the tensor core computes
            // those while the elementwise threads still work on tile t
            auto finish = [&](uint32_t t, int i, int hi, int r) -> bool {
                const int st = t % QS;
                if (!wait_quick(&ctl->p_full, t & 1, p.err, abort_flag)) return false;
                // accumulators of the previous head / item have been read
                if (i == 0 && nh > 0 && !wait_quick(&ctl->acc_free, (nh - 1) & 1, p.err, abort_flag)) return false;
                if (i == 0 && hi == 0 && r > 0 && !wait_quick(&ctl->k2_free, (r - 1) & 1, p.err, abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t sq = q0a + st * LY::QST_BYTES;
                issue_ss64<kDV>(tmem + tdV, wa, sq + 2 * LY::Q_BYTES, i > 0);                     // dV += W dO
                issue_ss64<kD>(tmem + tdK1, wa + LY::W_BYTES, sq, i > 0);                         // dK1 += dS1 Q1
                issue_ss64<kD>(tmem + tdK2, wa + 2 * LY::W_BYTES, sq + LY::Q_BYTES, i > 0 || hi > 0);   // dK2 += dS2 Q2
                mma_commit(&ctl->q_empty[st]);
                mma_commit(&ctl->w_free);
                return true;
            };
            for (int r = 0; ok && kv_item(p, r, G, cid, b, g, k0, i0, nq); ++r) {
                if (!wait_quick(&ctl->g_full, r & 1, p.err, abort_flag)) break;
                for (int hi = 0; ok && hi < r_grp; ++hi) {
                    if (!wait_quick(&ctl->h_full, nh & 1, p.err, abort_flag)) { ok = false; break; }
                    for (int i = 0; i < nq; ++i) {
                        const int st = gq % QS;
                        if (!wait_quick(&ctl->q_full[st], (gq / QS) & 1, p.err, abort_flag)) { ok = false; break; }
                        // the previous tile's logits have been read into registers
                        if (gq > 0 && !wait_quick(&ctl->s_free, (gq - 1) & 1, p.err, abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t sq = q0a + st * LY::QST_BYTES;
                        issue_nt<kD>(tmem + tS1, k1a, sq);                         // S1^T = K1 Q1^T
                        issue_nt<kD>(tmem + tS2, k2a, sq + LY::Q_BYTES);           // S2^T = K2 Q2^T
                        issue_nt<kDV>(tmem + tdP, va, sq + 2 * LY::Q_BYTES);       // dP^T = V dO^T
                        mma_commit(&ctl->s_full);
                        if (i > 0 && !finish(gq - 1, i - 1, hi, r)) { ok = false; break; }
                        ++gq;
                    }
                    if (!ok || !finish(gq - 1, nq - 1, hi, r)) { ok = false; break; }
                    mma_commit(&ctl->acc_ready);
                    mma_commit(&ctl->h_empty);
                    ++nh;
                }
                if (!ok) break;
                mma_commit(&ctl->k2_ready);
                mma_commit(&ctl->g_empty);
            }
            mma_commit(&ctl->mma_idle);
            drain_wait(&ctl->mma_idle, 0, p.err);
        }
        __syncwarp();
    } else {
        const int grp = (warp - 2) / 4;             // query columns [16 grp, 16 grp + 16) of each tile
        const int quarter = warp % 4;
        const int row = quarter * 32 + lane;        // key within the tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        uint32_t gq = 0, nh = 0;
        int b, g, k0, i0, nq;
        bool ok = true;
        auto store16 = [&](float *dst, uint32_t taddr, float mul, bool kin) {
            uint32_t o[16];
            tmem_ld16(taddr, o);
            tmem_ld_wait_regs16(o);
            if (kin) {
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    reinterpret_cast<float4 *>(dst)[v4] =
                        make_float4(__uint_as_float(o[4 * v4]) * mul, __uint_as_float(o[4 * v4 + 1]) * mul,
                                    __uint_as_float(o[4 * v4 + 2]) * mul, __uint_as_float(o[4 * v4 + 3]) * mul);
            }
        };
        for (int r = 0; ok && kv_item(p, r, G, cid, b, g, k0, i0, nq); ++r) {
            const int key = k0 + row;
            const int wkey_last = k0 + quarter * 32 + 31;      // this warp's last key
            for (int hi = 0; ok && hi < r_grp; ++hi) {
                const int h = g * r_grp + hi;
                const float nlam = -p.lambda[h];
                for (int i = 0; i < nq; ++i) {
                    const int q0 = (i0 + i) * kN + grp * 16;     // this group's first query column
                    const int st = gq % QS;
                    // the stage's vectors were written by the copy engine: observe its barrier too
                    if (!wait_quick(&ctl->s_full, gq & 1, p.err, abort_flag)) ok = false;
                    if (!wait_quick(&ctl->q_full[st], (gq / QS) & 1, p.err, abort_flag)) ok = false;
                    tc_fence_after();
                    const uint32_t tcol = tmem + lane_off + grp * 16;
                    uint32_t s1[16], s2[16], dp[16];
                    tmem_ld16(tcol + tS1, s1);
                    tmem_ld16(tcol + tS2, s2);
                    tmem_ld16(tcol + tdP, dp);
                    tmem_ld_wait_regs16(s1);
                    reg_fence16(s2);
                    reg_fence16(dp);
                    tc_fence_before();
                    mbar_arrive(&ctl->s_free);                  // the next tile's logits may overwrite S
                    const float *vec = reinterpret_cast<const float *>(smem + LY::OFF_Q + st * LY::QST_BYTES +
                                                                       2 * LY::Q_BYTES + LY::DO_BYTES) + grp * 16;
                    // every (key, query) pair of this warp and group is visible: no per-element mask
                    const bool clean = q0 + 15 < p.L && wkey_last < p.L && (!p.causal || wkey_last <= q0);
                    uint32_t pw[8], pd1[8], pd2[8];
                    // W = a1 - lambda a2, dS1 = a1 (dP - D1), dS2 = -lambda a2 (dP - D2) for
                    // pairs of query columns in packed float32 arithmetic; the per-pair
                    // visibility test only in the masked instance
                    auto pairs = [&](auto masked) {
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const float p1a = fast_exp2(fmaf(__uint_as_float(s1[e]), sl2, -vec[e]));
                            const float p1b = fast_exp2(fmaf(__uint_as_float(s1[e + 1]), sl2, -vec[e + 1]));
                            float n2a = fast_exp2(fmaf(__uint_as_float(s2[e]), sl2, -vec[64 + e]));
                            float n2b = fast_exp2(fmaf(__uint_as_float(s2[e + 1]), sl2, -vec[64 + e + 1]));
                            fmul2(n2a, n2b, nlam, nlam);
                            float wa = p1a, wb = p1b;
                            fadd2(wa, wb, n2a, n2b);
                            float ta = __uint_as_float(dp[e]), tb = __uint_as_float(dp[e + 1]);
                            float ua = ta, ub = tb;
                            fsub2(ta, tb, vec[128 + e], vec[128 + e + 1]);
                            fsub2(ua, ub, vec[192 + e], vec[192 + e + 1]);
                            fmul2(ta, tb, p1a, p1b);
                            fmul2(ua, ub, n2a, n2b);
                            if constexpr (decltype(masked)::value) {
                                const int q = q0 + e;
                                const bool va = q < p.L && key < p.L && (!p.causal || key <= q);
                                const bool vb = q + 1 < p.L && key < p.L && (!p.causal || key <= q + 1);
                                wa = va ? wa : 0.f;
                                ta = va ? ta : 0.f;
                                ua = va ? ua : 0.f;
                                wb = vb ? wb : 0.f;
                                tb = vb ? tb : 0.f;
                                ub = vb ? ub : 0.f;
                            }
                            pw[e / 2] = pack_bf16x2(wa, wb);
                            pd1[e / 2] = pack_bf16x2(ta, tb);
                            pd2[e / 2] = pack_bf16x2(ua, ub);
                        }
                    };
                    if (clean)
                        pairs(std::false_type{});
                    else
                        pairs(std::true_type{});
                    // the previous tile's products have read W / dS1 / dS2
                    if (gq > 0 && !wait_quick(&ctl->w_free, (gq - 1) & 1, p.err, abort_flag)) ok = false;
                    // row `row` of each K-major tile: 16-byte chunks 2 grp and 2 grp + 1 (query
                    // columns 16 grp .. 16 grp + 15), 128-byte swizzle: chunk c at c ^ (row % 8)
                    uint8_t *wrow = smem + LY::OFF_W + row * 128;
                    const int c0 = ((2 * grp) ^ (row & 7)) * 16, c1 = ((2 * grp + 1) ^ (row & 7)) * 16;
                    *reinterpret_cast<uint4 *>(wrow + c0) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    *reinterpret_cast<uint4 *>(wrow + c1) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
                    *reinterpret_cast<uint4 *>(wrow + LY::W_BYTES + c0) = make_uint4(pd1[0], pd1[1], pd1[2], pd1[3]);
                    *reinterpret_cast<uint4 *>(wrow + LY::W_BYTES + c1) = make_uint4(pd1[4], pd1[5], pd1[6], pd1[7]);
                    *reinterpret_cast<uint4 *>(wrow + 2 * LY::W_BYTES + c0) = make_uint4(pd2[0], pd2[1], pd2[2], pd2[3]);
                    *reinterpret_cast<uint4 *>(wrow + 2 * LY::W_BYTES + c1) = make_uint4(pd2[4], pd2[5], pd2[6], pd2[7]);
                    fence_proxy_async_smem();                   // visible to the tensor core's reads
                    mbar_arrive(&ctl->p_full);
                    ++gq;
                }
                ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
                // ---- dV and dK1 of head h
                if (ok) ok = warp_wait(&ctl->acc_ready, nh & 1, p.err, abort_flag);
                tc_fence_after();
                if (ok) {
                    const bool kin = key < p.L;
                    const size_t kix = (static_cast<size_t>(b) * p.L + (kin ? key : 0)) * p.hs + h;
                    store16(p.dvo + kix * kDV + grp * 32, tmem + lane_off + tdV + grp * 32, 1.f, kin);
                    store16(p.dvo + kix * kDV + grp * 32 + 16, tmem + lane_off + tdV + grp * 32 + 16, 1.f, kin);
                    store16(p.dk1 + kix * kD + grp * 16, tmem + lane_off + tdK1 + grp * 16, p.scale, kin);
                }
                tc_fence_before();
                mbar_arrive(&ctl->acc_free);
                ++nh;
                if (bar_red_or(1, kEwKv, !ok || *abort_flag)) ok = false;
            }
            if (!ok) break;
            // ---- dK2 of the item (summed over the group's heads)
            ok = warp_wait(&ctl->k2_ready, r & 1, p.err, abort_flag);
            tc_fence_after();
            if (ok) {
                const bool kin = key < p.L;
                const size_t kix = (static_cast<size_t>(b) * p.L + (kin ? key : 0)) * p.hn + g;
                store16(p.dk2 + kix * kD + grp * 16, tmem + lane_off + tdK2 + grp * 16, p.scale, kin);
            }
            tc_fence_before();
            mbar_arrive(&ctl->k2_free);
            if (bar_red_or(1, kEwKv, !ok || *abort_flag)) break;
        }
        tmem_ld_wait();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ==================================================================== dQ ==
// Item = (128-row query tile, b, noise group g); inside: the group's r
// signal heads, each over the 64-key tiles the rows see.

struct QLayout {
    static constexpr int KS = 3;
    static constexpr int Q_BYTES = kBM * kD * 2;          // 16 KiB
    static constexpr int DO_BYTES = kBM * kDV * 2;        // 32 KiB
    static constexpr int K_BYTES = kN * kD * 2;           // 8 KiB
    static constexpr int V_BYTES = kN * kDV * 2;          // 16 KiB
    static constexpr int KST_BYTES = 2 * K_BYTES + V_BYTES;
    static constexpr int OFF_Q2 = 0, OFF_Q1 = Q_BYTES, OFF_DO = 2 * Q_BYTES;
    static constexpr int OFF_K = OFF_DO + DO_BYTES;
    static constexpr int TILES = OFF_K + KS * KST_BYTES;
};

struct QCtrl {
    uint64_t g_full, g_empty;          // Q2 of the item
    uint64_t h_full, h_empty;          // Q1 and dO of the current head
    uint64_t k_full[3], k_empty[3];
    uint64_t s_full[2], p_full[2];     // [S buffer]
    uint64_t acc_ready, acc_free;      // dQ1 of a head
    uint64_t q2_ready, q2_free;        // dQ2 of an item
    uint64_t mma_idle;
    uint32_t tmem_base;
    int abort_flag;
};

constexpr int q_smem_bytes() {
    return QLayout::TILES + static_cast<int>((sizeof(QCtrl) + 1023) / 1024) * 1024 + 1024;
}

__device__ __forceinline__ bool q_item(const BwdTcParams &p, int r, int G, int cid, int &b, int &g, int &q0,
                                       int &nkv) {
    const int nqt = (p.L + kBM - 1) / kBM;
    const int per = p.B * p.hn;
    const long long n = static_cast<long long>(nqt) * per;
    const int k = (r & 1) ? (G - 1 - cid) : cid;
    const long long idx = static_cast<long long>(r) * G + k;
    if (idx >= n) return false;
    const int i = static_cast<int>(idx);
    q0 = (nqt - 1 - i / per) * kBM;
    b = (i % per) / p.hn;
    g = (i % per) % p.hn;
    const int kv_end = p.causal ? min(p.L, q0 + kBM) : p.L;
    nkv = (kv_end + kN - 1) / kN;
    return true;
}

constexpr int kEwQ = 512;           // dQ elementwise threads: 16 warps, four 16-column groups
constexpr int kThrQ = 64 + kEwQ;

__global__ void __launch_bounds__(kThrQ, 1)
gda_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmQ2,
                  const __grid_constant__ CUtensorMap tmdO, const __grid_constant__ CUtensorMap tmK1,
                  const __grid_constant__ CUtensorMap tmK2, const __grid_constant__ CUtensorMap tmV,
                  const BwdTcParams p) {
    using LY = QLayout;
    constexpr int KS = LY::KS;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, offset from the shared array itself so that accesses stay in the
    // shared state space (32-bit addresses)
    uint8_t *smem = smem_raw + ((0u - smem_u32(smem_raw)) & 1023u);
    QCtrl *ctl = reinterpret_cast<QCtrl *>(smem + LY::TILES);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cid = blockIdx.x, G = gridDim.x;
    const int r_grp = p.hs / p.hn;
    const int heads = p.hs + p.hn;

    if (threadIdx.x == 0) {
        mbar_init(&ctl->g_full, 1);
        mbar_init(&ctl->g_empty, 1);
        mbar_init(&ctl->h_full, 1);
        mbar_init(&ctl->h_empty, 1);
        for (int s = 0; s < KS; ++s) {
            mbar_init(&ctl->k_full[s], 1);
            mbar_init(&ctl->k_empty[s], 1);
        }
        for (int bb = 0; bb < 2; ++bb) {
            mbar_init(&ctl->s_full[bb], 1);
            mbar_init(&ctl->p_full[bb], kEwQ);
        }
        mbar_init(&ctl->acc_ready, 1);
        mbar_init(&ctl->acc_free, kEwQ);
        mbar_init(&ctl->q2_ready, 1);
        mbar_init(&ctl->q2_free, kEwQ);
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
    griddep_wait();      // the previous kernel's outputs (launched as its programmatic dependent)
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;
    // TMEM: two S buffers of S1 | S2 | dP (64 columns each) at [0,192) and
    // [192,384) | dQ1 [384,448) | dQ2 [448,512).  The logits of tile j+2 are
    // computed while the elementwise threads work on tile j+1.
    constexpr uint32_t kSB = 192, tS1 = 0, tS2 = 64, tdP = 128, tdQ1 = 384, tdQ2 = 448;

    if (warp == 0) {
        if (elect_one()) {
            tma_prefetch_desc(&tmQ1);
            tma_prefetch_desc(&tmQ2);
            tma_prefetch_desc(&tmdO);
            tma_prefetch_desc(&tmK1);
            tma_prefetch_desc(&tmK2);
            tma_prefetch_desc(&tmV);
            uint32_t gk = 0, nh = 0;
            int ng = 0;
            bool ok = true;
            int b, g, q0, nkv;
            for (int r = 0; ok && q_item(p, r, G, cid, b, g, q0, nkv); ++r) {
                if (r > 0 && !wait_quick(&ctl->g_empty, (r - 1) & 1, p.err, abort_flag)) break;
                mbar_arrive_expect_tx(&ctl->g_full, LY::Q_BYTES);
                tma_load_4d(smem + LY::OFF_Q2, &tmQ2, &ctl->g_full, 0, g, q0, b);
                ++ng;
                for (int hi = 0; ok && hi < r_grp; ++hi) {
                    const int h = g * r_grp + hi;
                    if (nh > 0 && !wait_quick(&ctl->h_empty, (nh - 1) & 1, p.err, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&ctl->h_full, LY::Q_BYTES + LY::DO_BYTES);
                    tma_load_4d(smem + LY::OFF_Q1, &tmQ1, &ctl->h_full, 0, h, q0, b);
                    tma_load_4d(smem + LY::OFF_DO, &tmdO, &ctl->h_full, 0, h, q0, b);
                    tma_load_4d(smem + LY::OFF_DO + kBM * 128, &tmdO, &ctl->h_full, 64, h, q0, b);
                    ++nh;
                    for (int j = 0; j < nkv; ++j) {
                        const int st = gk % KS;
                        if (gk >= KS && !wait_quick(&ctl->k_empty[st], ((gk / KS) - 1) & 1, p.err, abort_flag)) {
                            ok = false;
                            break;
                        }
                        uint8_t *sb = smem + LY::OFF_K + st * LY::KST_BYTES;
                        mbar_arrive_expect_tx(&ctl->k_full[st], LY::KST_BYTES);
                        tma_load_4d(sb, &tmK1, &ctl->k_full[st], 0, h, j * kN, b);
                        tma_load_4d(sb + LY::K_BYTES, &tmK2, &ctl->k_full[st], 0, g, j * kN, b);
                        tma_load_4d(sb + 2 * LY::K_BYTES, &tmV, &ctl->k_full[st], 0, h, j * kN, b);
                        tma_load_4d(sb + 2 * LY::K_BYTES + kN * 128, &tmV, &ctl->k_full[st], 64, h, j * kN, b);
                        ++gk;
                    }
                }
            }
            if (ng > 0) drain_wait(&ctl->g_full, (ng - 1) & 1, p.err);
            if (nh > 0) drain_wait(&ctl->h_full, (nh - 1) & 1, p.err);
            for (uint32_t j = (gk > KS ? gk - KS : 0); j < gk; ++j)
                drain_wait(&ctl->k_full[j % KS], (j / KS) & 1, p.err);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (elect_one()) {
            const uint32_t q1a = smem_u32(smem + LY::OFF_Q1), q2a = smem_u32(smem + LY::OFF_Q2);
            const uint32_t doa = smem_u32(smem + LY::OFF_DO), k0a = smem_u32(smem + LY::OFF_K);
            uint32_t gk = 0, nh = 0;
            bool ok = true;
            int b, g, q0, nkv;
            for (int r = 0; ok && q_item(p, r, G, cid, b, g, q0, nkv); ++r) {
                if (!wait_quick(&ctl->g_full, r & 1, p.err, abort_flag)) break;
                for (int hi = 0; ok && hi < r_grp; ++hi) {
                    if (!wait_quick(&ctl->h_full, nh & 1, p.err, abort_flag)) { ok = false; break; }
                    // logits of tile t into S buffer (gk + t) & 1
                    auto issue_s = [&](int t) -> bool {
                        const uint32_t gt = gk + t;
                        const int st = gt % KS;
                        if (!wait_quick(&ctl->k_full[st], (gt / KS) & 1, p.err, abort_flag)) return false;
                        tc_fence_after();
                        const uint32_t sk = k0a + st * LY::KST_BYTES;
                        const uint32_t sb = tmem + (gt & 1) * kSB;
                        issue_nt<kD>(sb + tS1, q1a, sk);                           // S1 = Q1 K1^T
                        issue_nt<kD>(sb + tS2, q2a, sk + LY::K_BYTES);             // S2 = Q2 K2^T
                        issue_nt<kDV>(sb + tdP, doa, sk + 2 * LY::K_BYTES);        // dP = dO V^T
                        mma_commit(&ctl->s_full[gt & 1]);
                        return true;
                    };
                    for (int t = 0; ok && t < 2 && t < nkv; ++t) ok = issue_s(t);
                    for (int j = 0; ok && j < nkv; ++j) {
                        const uint32_t gj = gk + j;
                        const int st = gj % KS;
                        const int bb = gj & 1;
                        if (!wait_quick(&ctl->p_full[bb], (gj >> 1) & 1, p.err, abort_flag)) { ok = false; break; }
                        if (j == 0 && nh > 0 && !wait_quick(&ctl->acc_free, (nh - 1) & 1, p.err, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (j == 0 && hi == 0 && r > 0 && !wait_quick(&ctl->q2_free, (r - 1) & 1, p.err, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sk = k0a + st * LY::KST_BYTES;
                        const uint32_t sb = tmem + bb * kSB;
                        issue_ts64q<kD>(tmem + tdQ1, sb + tS1, sk, j > 0);                          // dQ1 += dS1 K1
                        issue_ts64q<kD>(tmem + tdQ2, sb + tS2, sk + LY::K_BYTES, j > 0 || hi > 0);  // dQ2 += dS2 K2
                        mma_commit(&ctl->k_empty[st]);
                        // the buffer just read by those products takes the logits of tile j + 2
                        if (j + 2 < nkv) ok = issue_s(j + 2);
                    }
                    gk += nkv;
                    if (!ok) break;
                    mma_commit(&ctl->acc_ready);
                    mma_commit(&ctl->h_empty);
                    ++nh;
                }
                if (!ok) break;
                mma_commit(&ctl->q2_ready);
                mma_commit(&ctl->g_empty);
            }
            mma_commit(&ctl->mma_idle);
            drain_wait(&ctl->mma_idle, 0, p.err);
        }
        __syncwarp();
    } else {
        const int grp = (warp - 2) / 4;             // key columns [16 grp, 16 grp + 16) of each tile
        const int quarter = warp % 4;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        uint32_t gk = 0, nh = 0;
        int b, g, q0, nkv;
        bool ok = true;
        auto store16 = [&](float *dst, uint32_t taddr, bool in) {
            uint32_t o[16];
            tmem_ld16(taddr, o);
            tmem_ld_wait_regs16(o);
            if (in) {
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    reinterpret_cast<float4 *>(dst)[v4] =
                        make_float4(__uint_as_float(o[4 * v4]) * p.scale, __uint_as_float(o[4 * v4 + 1]) * p.scale,
                                    __uint_as_float(o[4 * v4 + 2]) * p.scale, __uint_as_float(o[4 * v4 + 3]) * p.scale);
            }
        };
        for (int r = 0; ok && q_item(p, r, G, cid, b, g, q0, nkv); ++r) {
            const int qrow = q0 + row;
            const bool in = qrow < p.L;
            const int last_key = p.causal ? min(qrow, p.L - 1) : p.L - 1;
            const int wrow_first = q0 + quarter * 32;   // this warp's first query row
            for (int hi = 0; ok && hi < r_grp; ++hi) {
                const int h = g * r_grp + hi;
                const float nlam = -p.lambda[h];
                const float nlse1 = in ? -p.lse[(static_cast<size_t>(b) * heads + h) * p.Lp + qrow] : 0.f;
                const float nlse2 = in ? -p.lse[(static_cast<size_t>(b) * heads + p.hs + g) * p.Lp + qrow] : 0.f;
                const float D1 = in ? p.D1[(static_cast<size_t>(b) * p.hs + h) * p.Lp + qrow] : 0.f;
                const float D2 = in ? p.D2[(static_cast<size_t>(b) * p.hs + h) * p.Lp + qrow] : 0.f;
                for (int j = 0; j < nkv; ++j) {
                    const uint32_t sb = tmem + lane_off + (gk & 1) * kSB + grp * 16;
                    if (!wait_quick(&ctl->s_full[gk & 1], (gk >> 1) & 1, p.err, abort_flag)) ok = false;
                    tc_fence_after();
                    uint32_t s1[16], s2[16], dp[16];
                    tmem_ld16(sb + tS1, s1);
                    tmem_ld16(sb + tS2, s2);
                    tmem_ld16(sb + tdP, dp);
                    tmem_ld_wait_regs16(s1);
                    reg_fence16(s2);
                    reg_fence16(dp);
                    const int kc0 = j * kN + grp * 16;
                    // every (query, key) pair of this warp and group is visible: no per-element mask
                    const bool clean = wrow_first + 31 < p.L && kc0 + 15 < p.L && (!p.causal || kc0 + 15 <= wrow_first);
                    uint32_t pd1[8], pd2[8];
                    // dS1 = a1 (dP - D1), dS2 = -lambda a2 (dP - D2) for pairs of key columns in
                    // packed float32 arithmetic; the visibility test only in the masked instance
                    auto pairs = [&](auto masked) {
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const float p1a = fast_exp2(fmaf(__uint_as_float(s1[e]), sl2, nlse1));
                            const float p1b = fast_exp2(fmaf(__uint_as_float(s1[e + 1]), sl2, nlse1));
                            float n2a = fast_exp2(fmaf(__uint_as_float(s2[e]), sl2, nlse2));
                            float n2b = fast_exp2(fmaf(__uint_as_float(s2[e + 1]), sl2, nlse2));
                            fmul2(n2a, n2b, nlam, nlam);
                            float ta = __uint_as_float(dp[e]), tb = __uint_as_float(dp[e + 1]);
                            float ua = ta, ub = tb;
                            fsub2(ta, tb, D1, D1);
                            fsub2(ua, ub, D2, D2);
                            fmul2(ta, tb, p1a, p1b);
                            fmul2(ua, ub, n2a, n2b);
                            if constexpr (decltype(masked)::value) {
                                const bool va = in && kc0 + e <= last_key;
                                const bool vb = in && kc0 + e + 1 <= last_key;
                                ta = va ? ta : 0.f;
                                ua = va ? ua : 0.f;
                                tb = vb ? tb : 0.f;
                                ub = vb ? ub : 0.f;
                            }
                            pd1[e / 2] = pack_bf16x2(ta, tb);
                            pd2[e / 2] = pack_bf16x2(ua, ub);
                        }
                    };
                    if (clean)
                        pairs(std::false_type{});
                    else
                        pairs(std::true_type{});
                    tmem_st8(sb + tS1, pd1);
                    tmem_st8(sb + tS2, pd2);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&ctl->p_full[gk & 1]);
                    ++gk;
                }
                ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
                if (ok) ok = warp_wait(&ctl->acc_ready, nh & 1, p.err, abort_flag);
                tc_fence_after();
                if (ok)
                    store16(p.dq1 + ((static_cast<size_t>(b) * p.L + (in ? qrow : 0)) * p.hs + h) * kD + grp * 16,
                            tmem + lane_off + tdQ1 + grp * 16, in);
                tc_fence_before();
                mbar_arrive(&ctl->acc_free);
                ++nh;
                if (bar_red_or(1, kEwQ, !ok || *abort_flag)) ok = false;
            }
            if (!ok) break;
            ok = warp_wait(&ctl->q2_ready, r & 1, p.err, abort_flag);
            tc_fence_after();
            if (ok)
                store16(p.dq2 + ((static_cast<size_t>(b) * p.L + (in ? qrow : 0)) * p.hn + g) * kD + grp * 16,
                        tmem + lane_off + tdQ2 + grp * 16, in);
            tc_fence_before();
            mbar_arrive(&ctl->q2_free);
            if (bar_red_or(1, kEwQ, !ok || *abort_flag)) break;
        }
        tmem_ld_wait();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// dlambda_h = -sum over (b, rows < L) of D2, in a fixed order
__global__ void __launch_bounds__(256) gda_bwd_dlambda_kernel(const BwdTcParams p) {
    griddep_wait();
    __shared__ float red[256];
    const int h = blockIdx.x;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // eight loads in flight per thread
    for (int b = 0; b < p.B; ++b) {
        const float *row = p.D2 + (static_cast<size_t>(b) * p.hs + h) * p.Lp;
        for (int i0 = 0; i0 < p.L; i0 += 8 * 256) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * 256 + static_cast<int>(threadIdx.x);
                if (i < p.L) acc[u] += row[i];
            }
        }
    }
    red[threadIdx.x] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
        if (static_cast<int>(threadIdx.x) < s) red[threadIdx.x] += red[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) p.dlambda[h] = -red[0];
}

bool map4(CUtensorMap *m, const void *base, uint64_t inner, uint64_t heads, uint64_t L, uint64_t B,
          uint32_t box_rows) {
    const uint64_t dims[4] = {inner, heads, L, B};
    const uint64_t str[3] = {inner * 2, heads * inner * 2, L * heads * inner * 2};
    const uint32_t box[4] = {64, 1, box_rows, 1};
    return encode_tmap_4d_bf16(m, base, dims, str, box);
}

}  // namespace

size_t backward_tc_workspace_bytes(int B, int L, int hs, int hn, int dv) {
    const size_t Lp = (static_cast<size_t>(L) + kBM - 1) / kBM * kBM;
    const size_t lse = sizeof(float) * B * static_cast<size_t>(hs + hn) * Lp;
    const size_t dvec = 2 * sizeof(float) * B * static_cast<size_t>(hs) * Lp;
    const size_t dO = 2 * static_cast<size_t>(B) * L * hs * dv;
    return lse + dvec + ((dO + 255) / 256) * 256 + 256;
}

int launch_backward_tc(const BackwardTcArgs &a, cudaStream_t stream) {
    if (a.d != kD || a.dv != kDV) return GDA_ERR_UNSUPPORTED;
    const int Lp = (a.L + kBM - 1) / kBM * kBM;
    uint8_t *w = static_cast<uint8_t *>(a.workspace);
    float *lse = reinterpret_cast<float *>(w);
    float *D1 = lse + static_cast<size_t>(a.B) * (a.hs + a.hn) * Lp;
    float *D2 = D1 + static_cast<size_t>(a.B) * a.hs * Lp;
    __nv_bfloat16 *dO = reinterpret_cast<__nv_bfloat16 *>(D2 + static_cast<size_t>(a.B) * a.hs * Lp);

    // pass 1: the statistics
    PrefillArgs pa{a.q1, a.k1, a.q2, a.k2, a.v, a.lambda, a.lambda_init, nullptr, a.B, a.L, a.hs, a.hn,
                   a.d, a.dv, a.causal, a.eps, a.flags, a.dev_err};
    int st = launch_lse_pass(pa, lse, Lp, stream);
    if (st != GDA_OK) return st;

    BwdTcParams p;
    p.lambda = a.lambda;
    p.lse = lse;
    p.dy = static_cast<const __nv_bfloat16 *>(a.dy);
    p.dO = dO;
    p.D1 = D1;
    p.D2 = D2;
    p.dq1 = a.dq1;
    p.dk1 = a.dk1;
    p.dq2 = a.dq2;
    p.dk2 = a.dk2;
    p.dvo = a.dv_out;
    p.dlambda = a.dlambda;
    p.err = a.dev_err;
    p.lambda_init = a.lambda_init;
    p.eps = a.eps;
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a.d)));
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.d)));
    p.B = a.B;
    p.L = a.L;
    p.Lp = Lp;
    p.hs = a.hs;
    p.hn = a.hn;
    p.causal = a.causal;
    p.no_norm = (a.flags & GDA_FLAG_NO_NORM) ? 1 : 0;

    const uint64_t B = a.B, L = a.L, hs = a.hs, hn = a.hn;
    CUtensorMap q1_128, q1_64, k1_128, k1_64, q2_128, q2_64, k2_128, k2_64, v_128, v_64, do_128, do_64;
    if (!map4(&q1_128, a.q1, kD, hs, L, B, 128) || !map4(&q1_64, a.q1, kD, hs, L, B, 64) ||
        !map4(&k1_128, a.k1, kD, hs, L, B, 128) || !map4(&k1_64, a.k1, kD, hs, L, B, 64) ||
        !map4(&q2_128, a.q2, kD, hn, L, B, 128) || !map4(&q2_64, a.q2, kD, hn, L, B, 64) ||
        !map4(&k2_128, a.k2, kD, hn, L, B, 128) || !map4(&k2_64, a.k2, kD, hn, L, B, 64) ||
        !map4(&v_128, a.v, kDV, hs, L, B, 128) || !map4(&v_64, a.v, kDV, hs, L, B, 64) ||
        !map4(&do_128, dO, kDV, hs, L, B, 128) || !map4(&do_64, dO, kDV, hs, L, B, 64))
        return GDA_ERR_CUDA;

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    const long long nqt = (a.L + kBM - 1) / kBM;

    constexpr int smem_p = prep_smem_bytes();
    constexpr int smem_kv = kv_smem_bytes();
    constexpr int smem_q = q_smem_bytes();
    static_assert(smem_p <= 232448 && smem_kv <= 232448 && smem_q <= 232448, "shared memory budget");
    e = cudaFuncSetAttribute(gda_bwd_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_p);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gda_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gda_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q);
    if (e != cudaSuccess) return record_cuda_error(e);

    long long gp = nqt * a.B * a.hs;
    if (gp > sms) gp = sms;
    e = launch_dependent(gda_bwd_prep_kernel, static_cast<unsigned>(gp), kThrP, smem_p, stream, q1_128, k1_64,
                         q2_128, k2_64, v_64, p);
    long long gkv = nqt * a.B * a.hn;
    if (gkv > sms) gkv = sms;
    if (e == cudaSuccess)
        e = launch_dependent(gda_bwd_dkdv_kernel, static_cast<unsigned>(gkv), kThrKv, smem_kv, stream, k1_128,
                             k2_128, v_128, q1_64, q2_64, do_64, p);
    if (e == cudaSuccess)
        e = launch_dependent(gda_bwd_dq_kernel, static_cast<unsigned>(gkv), kThrQ, smem_q, stream, q1_128, q2_128,
                             do_128, k1_64, k2_64, v_64, p);
    if (e == cudaSuccess) e = launch_dependent(gda_bwd_dlambda_kernel, a.hs, 256, 0, stream, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

}  // namespace gda
