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
// runs two sweeps over its visible keys (128-key tiles), both in one CTA:
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
// epilogue only applies the headwise norm.  Forming P_h in float32 before its
// one rounding keeps the rounding error relative to the difference map, not
// to its two terms.  No statistics leave the SM: no workspace.
//
// Throughput facts this layout follows (tcgen05.mma with M = 128, K = 64,
// measured on GB300): an N = 64 logit product takes as long as an N = 128
// one (about 367 cycles), and a value product reading P from shared memory
// (313 cycles at N = 128) is faster than one reading it from TMEM (439).
//
// TMEM (512 columns): accumulators O_h at [128 h, 128 h + 128) for h < S,
// then NB = 4 - S slots of 128 columns for 128-key logit tiles (one at S = 3);
// phase A also uses the accumulator columns as logit slots.  A slot is released
// as soon as the compute warps have loaded its tile into registers (P goes to
// shared memory).
// Warp roles (persistent CTA, one per SM, 20 warps):
//   warp 0      TMA producer: Q2 and the S Q1 tiles once per item, then one ring
//               of 16 KB slots carrying 128-key K tiles and 64-key V tiles in
//               exactly the order the MMAs consume them;
//   warp 1      TMEM allocator and logit-MMA issuer (SS, K-major, N = 128);
//   warp 2      value-MMA issuer (SS: P from shared memory, V as an MN-major
//               operand), LAG uses behind the logits; the two issuers sit on
//               different SM sub-partitions and each skips the other's ring
//               entries;
//   warp 3      idle (completes the first warpgroup, which hands registers to
//               the compute warpgroups with setmaxnreg);
//   warps 4-19  compute (thread = query row = TMEM lane; warp w takes keys
//               [32 k, 32 k + 32) of each tile, k = (w - 4) / 4: four compute
//               warps per SM sub-partition): statistics, P, and the epilogue.
// Short items (at most kStageOutTiles key tiles) stage the output rows in the P
// buffers and write them with TMA stores (one thread per row quarter) and keep the
// statistics sweep's map loop rolled; longer items, where the epilogue is a small
// share, store each thread's row segment and unroll that loop.
// Every mbarrier wait is bounded (1 s) and sets GDA_DEVERR_PREFILL_TIMEOUT.
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

constexpr int kGBN = 128;              // keys per logit tile
constexpr int kStageOutTiles = 28;     // longest item (key tiles) that takes the short-item instance
constexpr int kPH = 64;                // keys per P half / V tile
#ifndef GDA_GROUP_KEYS_PER_THREAD
#define GDA_GROUP_KEYS_PER_THREAD 32
#endif
constexpr int kKQ = GDA_GROUP_KEYS_PER_THREAD;   // keys of a 128-key tile per compute thread
constexpr int kNQ = kGBN / kKQ;                  // compute threads per query row
constexpr int kGComputeWarps = 4 * kNQ;
// warps 0-3: TMA producer (0), logit MMA issuer (1), value MMA issuer (2), one idle; warps
// 4..: compute.  The first warpgroup hands registers to the compute warpgroups (setmaxnreg).
// With 16 compute warps, 640 threads launch with 96 registers each (the most five warps per
// SM sub-partition allow): 4 x 32 x 32 + 16 x 32 x 112 = 640 x 96.  With 8 compute warps,
// 384 threads launch with 168: 4 x 32 x 40 + 8 x 32 x 232 <= 384 x 168.
constexpr int kGCtrlWarps = 4;
constexpr int kGThreads = 32 * (kGCtrlWarps + kGComputeWarps);
constexpr int kGLaunchRegs = kGComputeWarps == 16 ? 96 : 168;
constexpr int kGCtrlRegs = kGComputeWarps == 16 ? 32 : 40;
constexpr int kGComputeRegs = kGComputeWarps == 16 ? 112 : 232;
static_assert(kGCtrlRegs * 32 * kGCtrlWarps + kGComputeRegs * 32 * kGComputeWarps <= kGLaunchRegs * kGThreads,
              "register split exceeds the launch pool");
static_assert(kKQ == 32 || kKQ == 64, "a thread takes 32 or 64 keys of each tile");

template <int S> struct GLayout {
    // TMEM: four 128-column slots; slot h < S holds O_h.  Phase A (statistics)
    // uses all four slots for logit tiles (the accumulators are free until the
    // item's first value MMA), phase B the NB slots above the accumulators.
    static constexpr int NB = 4 - S;                     // phase-B logit slots
    static constexpr int LAG = NB + 1;                   // value MMA of use u issued after logit MMA of u + LAG
    static constexpr int NR = 6;                         // ring of 16 KB K / V tiles
    static constexpr int Q_BYTES = kBM * 64 * 2;         // one head's 128 x 64 query tile
    static constexpr int R_BYTES = 16384;                // ring slot: a 128 x 64 K tile or a 64 x 128 V tile
    static constexpr int PH_BYTES = kBM * kPH * 2;       // one 128 x 64 bf16 half of a P tile
    static constexpr int OFF_Q = 0;                      // Q2, then Q1 of heads h0 .. h0+S-1
    static constexpr int OFF_R = OFF_Q + (S + 1) * Q_BYTES;
    static constexpr int OFF_P = OFF_R + NR * R_BYTES;   // P tiles [buffer][half: keys 0-63, 64-127]
    static constexpr int TILES = OFF_P + 4 * PH_BYTES;
    static_assert(NB >= 1, "TMEM budget");
    static_assert(kGBN * 64 * 2 == R_BYTES && kPH * 128 * 2 == R_BYTES, "ring slot size");
};

// Physical TMEM slot of phase-A use a of an item: the phase-B slots first (no
// wait for the previous item's epilogue), then the accumulator slots.
template <int S>
__device__ __forceinline__ uint32_t slot_a(uint32_t a) {
    const uint32_t k = a % 4;
    return k < static_cast<uint32_t>(4 - S) ? S + k : k - (4 - S);
}

// Post-increment of counter number `slot` of four (kept in registers).
__device__ __forceinline__ uint32_t bump(uint32_t (&cnt)[4], uint32_t slot) {
    uint32_t k = 0;
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q)
        if (q == slot) {
            k = cnt[q];
            cnt[q] = k + 1;
        }
    return k;
}

struct GCtrl {
    uint64_t q_full, q_empty;
    uint64_t r_full[6], r_empty[6];      // K / V ring
    uint64_t s_full[4], s_free[4];       // TMEM logit slots
    uint64_t p_full[2][2], p_empty[2][2];   // [P buffer][half]
    uint64_t o_final, o_free, mma_idle;
    uint32_t tmem_base;
    int abort_flag;
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

// Shared-memory matrix descriptor (128-byte swizzle) as two words: the low word holds
// the start address and the leading byte offset, the high word the stride byte offset,
// the descriptor version and the layout.  Advancing the start by b bytes (b a multiple
// of 16, the tile inside shared memory) adds b / 16 to the low word.
__host__ __device__ constexpr uint32_t sw128_desc_hi(uint32_t sbo) {
    return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ __forceinline__ uint32_t sw128_desc_lo(uint32_t addr, uint32_t lbo) {
    return ((addr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ uint64_t desc_words(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}

// Position in the K / V ring: slot and the parity of its fill.
template <int NR>
struct RingPos {
    uint32_t st = 0, ph = 0;
    __device__ __forceinline__ void advance(uint32_t n) {
        st += n;
        while (st >= static_cast<uint32_t>(NR)) {
            st -= NR;
            ph ^= 1u;
        }
    }
};

template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Every lane of the warp arrives once (the barriers the compute warps release count
// lanes): no warp-level synchronisation and no single-lane branch on the hot path.
__device__ __forceinline__ void lanes_arrive(uint64_t *bar) { mbar_arrive(bar); }

// Bounded wait that first polls once without the suspend-time hint (a wait whose phase
// has already completed costs about a third as much as the hinted form), then takes the
// bounded hinted wait.
__device__ __forceinline__ bool wait_fast(uint64_t *bar, uint32_t parity, unsigned *err, volatile int *abort) {
    const uint32_t a = smem_u32(bar);
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
    return mbar_wait(bar, parity, err, GDA_DEVERR_PREFILL_TIMEOUT, abort);
}

// Bounded wait that polls without the suspend hint for up to 256 tries before falling back
// to the hinted wait: the issuers' waits on the phase-B chain (a logit slot freed, a P tile
// written) usually end within that window, and the hinted wait's wake-up would delay the
// next MMA (7.41 -> 7.05 ms on the 3:1 L = 32768 workload; spinning on every issuer wait
// instead steals issue slots from the compute warps and costs 12 %).
__device__ __forceinline__ bool wait_spin(uint64_t *bar, uint32_t parity, unsigned *err, volatile int *abort) {
    const uint32_t a = smem_u32(bar);
    for (uint32_t it = 0; it < 256u; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return mbar_wait(bar, parity, err, GDA_DEVERR_PREFILL_TIMEOUT, abort);
}

__device__ __forceinline__ bool warp_wait_fast(uint64_t *bar, uint32_t parity, unsigned *err, volatile int *abort) {
    return __all_sync(0xffffffffu, wait_fast(bar, parity, err, abort));
}

template <int S, bool kStageOut>
__global__ void __launch_bounds__(kGThreads, 1)
gda_prefill_group_kernel(const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmK1,
                         const __grid_constant__ CUtensorMap tmQ2, const __grid_constant__ CUtensorMap tmK2,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                         const GParams p) {
    using LY = GLayout<S>;
    constexpr int NB = LY::NB, LAG = LY::LAG, NR = LY::NR;
    constexpr int M = S + 1;                 // maps per item: noise map (0), signal heads (1..S)
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned; offsetting the shared array itself (no integer round trip) keeps
    // every access below in the shared state space (32-bit addresses, LDS / STS)
    uint8_t *smem = smem_raw + ((0u - smem_u32(smem_raw)) & 1023u);
    GCtrl *ctl = reinterpret_cast<GCtrl *>(smem + LY::TILES);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int cid = blockIdx.x;
    const int G = gridDim.x;

    if (threadIdx.x == 0) {
        mbar_init(&ctl->q_full, 1);
        mbar_init(&ctl->q_empty, 1);
        for (int s = 0; s < NR; ++s) {
            mbar_init(&ctl->r_full[s], 1);
            mbar_init(&ctl->r_empty[s], 1);
        }
        for (int s = 0; s < 4; ++s) {
            mbar_init(&ctl->s_full[s], 1);
            mbar_init(&ctl->s_free[s], 32 * kGComputeWarps);
        }
        for (int s = 0; s < 2; ++s)
            for (int hf = 0; hf < 2; ++hf) {
                mbar_init(&ctl->p_full[s][hf], 16 * kGComputeWarps);     // the lanes writing the half
                mbar_init(&ctl->p_empty[s][hf], 1);
            }
        mbar_init(&ctl->o_final, 1);
        mbar_init(&ctl->o_free, 32 * kGComputeWarps);
        mbar_init(&ctl->mma_idle, 2);                              // one commit per MMA issuer
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

    if (warp < kGCtrlWarps) {
      regs_dec<kGCtrlRegs>();
      if (warp == 0) {
        // ================================================= TMA producer
        if (elect_one()) {
            tma_prefetch_desc(&tmQ1);
            tma_prefetch_desc(&tmK1);
            tma_prefetch_desc(&tmQ2);
            tma_prefetch_desc(&tmK2);
            tma_prefetch_desc(&tmV);
            if constexpr (kStageOut) tma_prefetch_desc(&tmO);
            uint32_t ct = 0;
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
                // next ring slot (K and V tiles share one ring, filled in consumption order)
                auto ring = [&](uint32_t bytes) -> uint8_t * {
                    const int st = ct % NR;
                    if (ct >= NR && !wait_bar(&ctl->r_empty[st], ((ct / NR) - 1) & 1, p.err, abort_flag))
                        return nullptr;
                    mbar_arrive_expect_tx(&ctl->r_full[st], bytes);
                    return smem + LY::OFF_R + st * LY::R_BYTES;
                };
                // 128-key K tile of map m (0: noise head g, 1..S: signal head h0 + m - 1) at key tile j
                auto load_k = [&](int m, int j) -> bool {
                    uint8_t *dst = ring(LY::R_BYTES);
                    if (!dst) return false;
                    uint64_t *bar = &ctl->r_full[ct % NR];
                    if (m == 0)
                        tma_load_4d(dst, &tmK2, bar, 0, it.g, j * kGBN, it.b);
                    else
                        tma_load_4d(dst, &tmK1, bar, 0, it.h0 + m - 1, j * kGBN, it.b);
                    ++ct;
                    return true;
                };
                // 64-key V tile of signal head h0 + h, keys j * 128 + half * 64 ..
                auto load_v = [&](int h, int j, int half) -> bool {
                    uint8_t *dst = ring(LY::R_BYTES);
                    if (!dst) return false;
                    uint64_t *bar = &ctl->r_full[ct % NR];
                    const int key0 = j * kGBN + half * kPH;
                    tma_load_4d(dst, &tmV, bar, 0, it.h0 + h, key0, it.b);
                    tma_load_4d(dst + kPH * 128, &tmV, bar, 64, it.h0 + h, key0, it.b);
                    ++ct;
                    return true;
                };
                // phase A: every map's K tiles, key tile by key tile
                for (int j = 0; ok && j < it.nkv; ++j)
                    for (int m = 0; ok && m < M; ++m) ok = load_k(m, j);
                // phase B: the same K tiles again, with each P-use's two V tiles LAG uses later
                const int nB = it.nkv * M;
                for (int i = 0; ok && i < nB; ++i) {
                    ok = load_k(i % M, i / M);
                    if (ok && i >= LAG && (i - LAG) % M != 0) {
                        const int v = i - LAG;
                        ok = load_v(v % M - 1, v / M, 0) && load_v(v % M - 1, v / M, 1);
                    }
                }
                for (int v = (nB > LAG ? nB - LAG : 0); ok && v < nB; ++v)
                    if (v % M != 0) ok = load_v(v % M - 1, v / M, 0) && load_v(v % M - 1, v / M, 1);
            }
            // our own copies must land before the CTA may exit
            if (nq > 0) drain_wait(&ctl->q_full, (nq - 1) & 1, p.err);
            for (uint32_t j = (ct > NR ? ct - NR : 0); j < ct; ++j)
                drain_wait(&ctl->r_full[j % NR], (j / NR) & 1, p.err);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================= logit MMA issuer
        if (elect_one()) {
            const uint32_t qlo0 = sw128_desc_lo(smem_u32(smem + LY::OFF_Q), 16);
            const uint32_t klo0 = sw128_desc_lo(smem_u32(smem + LY::OFF_R), 16);
            constexpr uint32_t hi_k = sw128_desc_hi(1024);
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kGBN, 0);
            uint32_t cnt[4] = {0, 0, 0, 0};    // uses of each TMEM slot so far
            RingPos<NR> rp;
            bool ok = true;
            GItem it;
            int nitem = 0;
            bool o_ready = true;
            // the accumulator slots are free once the previous item's epilogue has read them
            auto need_o = [&]() -> bool {
                if (o_ready) return true;
                o_ready = true;
                return nitem == 0 || wait_fast(&ctl->o_free, (nitem - 1) & 1, p.err, abort_flag);
            };
            // logit MMA of map m into TMEM slot `slot`: 128 x 128 x 64 as four K = 16 steps
            // (`spin`: the phase-B chain, where the slot's release is waited for by spinning)
            auto qk = [&](int m, uint32_t slot, bool spin) -> bool {
                const uint32_t k = bump(cnt, slot);
                if (slot < static_cast<uint32_t>(S) && !need_o()) return false;
                // the K tile is nearly always in the ring by now: its wait comes first, so that
                // only the slot's release stands between that release and the MMA
                if (!wait_fast(&ctl->r_full[rp.st], rp.ph, p.err, abort_flag)) return false;
                if (k >= 1 && !(spin ? wait_spin(&ctl->s_free[slot], (k - 1) & 1, p.err, abort_flag)
                                     : wait_fast(&ctl->s_free[slot], (k - 1) & 1, p.err, abort_flag)))
                    return false;
                tc_fence_after();
                const uint32_t qlo = qlo0 + m * (LY::Q_BYTES >> 4), klo = klo0 + rp.st * (LY::R_BYTES >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem + slot * 128, desc_words(qlo + 2 * kk, hi_k), desc_words(klo + 2 * kk, hi_k), idesc_qk,
                           kk > 0 ? 1u : 0u);
                mma_commit(&ctl->s_full[slot]);
                mma_commit(&ctl->r_empty[rp.st]);
                rp.advance(1);
                return true;
            };
            for (int rr = 0; ok && gitem_of(p, S, rr, G, cid, it); ++rr) {
                if (!wait_fast(&ctl->q_full, rr & 1, p.err, abort_flag)) break;
                o_ready = false;
                const int nA = it.nkv * M;
                for (int a = 0; ok && a < nA; ++a) ok = qk(a % M, slot_a<S>(a), false);
                const int nB = it.nkv * M;
                for (int i = 0; ok && i < nB; ++i) {
                    ok = qk(i % M, S + i % NB, true);
                    if (ok && i == nB - 1) mma_commit(&ctl->q_empty);     // the item's last logit MMA
                    if (i >= LAG && (i - LAG) % M != 0) rp.advance(2);     // the value issuer's two V tiles
                }
                for (int v = (nB > LAG ? nB - LAG : 0); v < nB; ++v)
                    if (v % M != 0) rp.advance(2);
                ++nitem;
            }
            // every issued MMA completes before TMEM is released
            mma_commit(&ctl->mma_idle);
            drain_wait(&ctl->mma_idle, 0, p.err);
        }
        __syncwarp();
      } else if (warp == 2) {
        // ================================================= value MMA issuer
        if (elect_one()) {
            const uint32_t plo0 = sw128_desc_lo(smem_u32(smem + LY::OFF_P), 16);
            const uint32_t vlo0 = sw128_desc_lo(smem_u32(smem + LY::OFF_R), kPH * 128);
            constexpr uint32_t hi_pv = sw128_desc_hi(1024);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, 128, 1);
            uint32_t pk = 0;
            RingPos<NR> rp;
            bool ok = true;
            GItem it;
            int nitem = 0;
            bool o_ready = true;
            auto need_o = [&]() -> bool {
                if (o_ready) return true;
                o_ready = true;
                return nitem == 0 || wait_fast(&ctl->o_free, (nitem - 1) & 1, p.err, abort_flag);
            };
            // value MMAs of P-use v (phase-B index) of the current item: O_h += P_h V_h, one
            // MMA group per 64-key half
            auto pv = [&](int v) -> bool {
                const int h = v % (S + 1) - 1, j = v / (S + 1);
                const uint32_t pb = pk & 1;
                if (!need_o()) return false;
                for (int half = 0; half < 2; ++half) {
                    if (!wait_spin(&ctl->p_full[pb][half], (pk >> 1) & 1, p.err, abort_flag)) return false;
                    if (!wait_fast(&ctl->r_full[rp.st], rp.ph, p.err, abort_flag)) return false;
                    tc_fence_after();
                    const uint32_t plo = plo0 + (pb * 2 + half) * (LY::PH_BYTES >> 4);
                    const uint32_t vlo = vlo0 + rp.st * (LY::R_BYTES >> 4);
#pragma unroll
                    for (int k = 0; k < kPH / 16; ++k)
                        mma_ss(tmem + 128 * h, desc_words(plo + 2 * k, hi_pv), desc_words(vlo + 128 * k, hi_pv), idesc_pv,
                               (j > 0 || half > 0 || k > 0) ? 1u : 0u);
                    mma_commit(&ctl->p_empty[pb][half]);
                    mma_commit(&ctl->r_empty[rp.st]);
                    rp.advance(1);
                }
                ++pk;
                return true;
            };
            for (int rr = 0; ok && gitem_of(p, S, rr, G, cid, it); ++rr) {
                o_ready = false;
                const int nA = it.nkv * M;
                rp.advance(nA);                                          // the phase-A K tiles
                const int nB = it.nkv * M;
                for (int i = 0; ok && i < nB; ++i) {
                    rp.advance(1);                                       // K tile of logit use i
                    if (i >= LAG && (i - LAG) % M != 0) ok = pv(i - LAG);
                }
                for (int v = (nB > LAG ? nB - LAG : 0); ok && v < nB; ++v)
                    if (v % M != 0) ok = pv(v);
                if (!ok) break;
                mma_commit(&ctl->o_final);
                ++nitem;
            }
            mma_commit(&ctl->mma_idle);
            drain_wait(&ctl->mma_idle, 0, p.err);
        }
        __syncwarp();
      }
    } else {
        // ================================================= compute warps
        regs_inc<kGComputeRegs>();
        const int kq = (warp - kGCtrlWarps) / 4;  // keys [kKQ kq, kKQ kq + kKQ) of every 128-key tile
        const int half = (kq * kKQ) / kPH;        // the P half (value MMA) those keys belong to
        const int quarter = warp % 4;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t row_bar = 1 + quarter;     // the kNQ warps that hold this row's key parts
        constexpr uint32_t kRowThreads = 32 * kNQ;
        const float sl2 = p.scale_log2;
        // this thread's 16-byte chunks of its row in its P half (buffer 0)
        uint8_t *pbuf0 = smem + LY::OFF_P + half * LY::PH_BYTES + row * 128;
        const int chunk0 = ((kq * kKQ) % kPH) / 8;
        // Per-item exchange between the kNQ warps that hold a row's key parts: 32 words in the
        // row's own 128 bytes of P buffer 0, half 0 (phase-A maximum and sum of each part and
        // map) and half 1 (epilogue sums of squares of each part and head).  Only the warps of
        // the row's quarter touch those bytes, and they are synchronised by the row barrier;
        // no value MMA reads them while the exchange is in use (before the item's first P tile
        // of the row, after its last value MMA).  Word e sits at (e + row) % 32, so a warp's 32
        // rows fall into 32 banks.
        static_assert(kNQ * 8 <= 32 && kNQ * 4 <= 32 && kGBN == kBM, "exchange layout");
        float *const xrow_a = reinterpret_cast<float *>(smem + LY::OFF_P + row * 128);
        float *const xrow_b = reinterpret_cast<float *>(smem + LY::OFF_P + LY::PH_BYTES + row * 128);
        auto xslot = [&](float *base, int e) -> float & { return base[(e + row) & 31]; };
        uint32_t cnt[4] = {0, 0, 0, 0};    // uses of each TMEM slot so far
        uint32_t pk = 0;
        GItem it;
        for (int rr = 0; gitem_of(p, S, rr, G, cid, it); ++rr) {
            const int qrow = it.q0 + row;
            const bool in = qrow < p.L;
            const int last_key = p.causal ? min(p.koff + qrow, p.Lk - 1) : p.Lk - 1;
            float lam[S];
#pragma unroll
            for (int h = 0; h < S; ++h) lam[h] = p.lambda[it.h0 + h];
            bool ok = true;

            // this thread's kKQ logits of TMEM slot `slot` into x
            auto read_slot = [&](uint32_t (&x)[kKQ], uint32_t slot) {
#pragma unroll
                for (int c = 0; c < kKQ / 32; ++c)
                    tmem_ld32(tmem + lane_off + slot * 128 + kq * kKQ + c * 32,
                              *reinterpret_cast<uint32_t(*)[32]>(&x[c * 32]));
                tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&x[0]));
                if constexpr (kKQ == 64) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&x[32]));
            };
            // wait for the logit MMA of the slot's next use, then read it
            auto acquire = [&](uint32_t (&x)[kKQ], uint32_t slot) {
                const uint32_t k = bump(cnt, slot);
                if (!wait_fast(&ctl->s_full[slot], k & 1, p.err, abort_flag)) ok = false;   // no vote: only sets the flag
                tc_fence_after();
                read_slot(x, slot);
            };
            auto release = [&](uint32_t slot) {
                tc_fence_before();
                lanes_arrive(&ctl->s_free[slot]);
            };
            auto load_use = [&](uint32_t (&x)[kKQ], uint32_t slot) {
                acquire(x, slot);
                release(slot);
            };
            // key tiles [0, jfull) hold no key past the last visible key of any row of this
            // warp (its first row has the smallest); only the tiles from jfull on take the
            // per-key compare
            const int min_last = p.causal ? min(p.koff + it.q0 + quarter * 32, p.Lk - 1) : p.Lk - 1;
            const int tfull = min_last - kq * kKQ - (kKQ - 1);
            const int jfull = tfull < 0 ? 0 : min(it.nkv, tfull / kGBN + 1);

            // ---------------------------------------------- phase A: row statistics
            // Each key quarter of the row keeps a reference mx and the sum ls of 2^(s c - mx).
            // The reference is the exact maximum of the first tile, floored at -1e30 so that a
            // quarter without a visible key sums zeros; later tiles exponentiate against it
            // directly, so no per-tile maximum sits on the critical path.  When a tile's sum
            // exceeds 2^16 (or is not finite) in any row of the warp, the warp reads the tile
            // from TMEM again (its slot is released only after the check), moves the reference
            // to the tile's maximum, rescales the running sum and sums the tile afresh.
            float mx[M], ls[M];
            auto tile_max = [&](const uint32_t (&x)[kKQ]) -> float {
                float m4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) m4[i] = __uint_as_float(x[i]);
#pragma unroll
                for (int e = 4; e + 8 <= kKQ; e += 8)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        m4[i] = max3f(m4[i], __uint_as_float(x[e + 2 * i]), __uint_as_float(x[e + 2 * i + 1]));
#pragma unroll
                for (int i = 0; i < 4; ++i) m4[i] = fmaxf(m4[i], __uint_as_float(x[kKQ - 4 + i]));
                return max3f(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2;
            };
            auto tile_sum = [&](const uint32_t (&x)[kKQ], float ref) -> float {
                const float neg = -ref;
                float sa = 0.f, sb = 0.f, sc = 0.f, sd = 0.f;
#pragma unroll
                for (int e = 0; e < kKQ; e += 4) {
                    float x0 = __uint_as_float(x[e]), x1 = __uint_as_float(x[e + 1]);
                    float x2 = __uint_as_float(x[e + 2]), x3 = __uint_as_float(x[e + 3]);
                    ffma2(x0, x1, sl2, sl2, neg, neg);
                    ffma2(x2, x3, sl2, sl2, neg, neg);
                    fadd2(sa, sb, fast_exp2(x0), fast_exp2(x1));
                    fadd2(sc, sd, fast_exp2(x2), fast_exp2(x3));
                }
                return (sa + sb) + (sc + sd);
            };
            auto mask_x = [&](uint32_t (&x)[kKQ], int k0) {
#pragma unroll
                for (int e = 0; e < kKQ; ++e)
                    if (k0 + e > last_key) x[e] = __float_as_uint(-INFINITY);
            };
            // map m of key tile j, with that map's running statistics (mxm, lsm); the unrolled
            // loop below spells the same steps out with the statistics indexed by map
            auto stats_map = [&](int j, int m, float &mxm, float &lsm, auto first, auto masked) {
                const int k0 = j * kGBN + kq * kKQ;
                const uint32_t slot = slot_a<S>(j * M + m);
                uint32_t x[kKQ];
                acquire(x, slot);
                if constexpr (decltype(masked)::value) mask_x(x, k0);
                if constexpr (decltype(first)::value) {
                    mxm = fmaxf(tile_max(x), -1e30f);
                    lsm = tile_sum(x, mxm);
                } else {
                    float ts = tile_sum(x, mxm);
                    if (__any_sync(0xffffffffu, !(ts <= 65536.f))) {
                        read_slot(x, slot);
                        if constexpr (decltype(masked)::value) mask_x(x, k0);
                        const float nr = fmaxf(mxm, tile_max(x));
                        lsm *= fast_exp2(mxm - nr);
                        mxm = nr;
                        ts = tile_sum(x, nr);
                    }
                    lsm += ts;
                }
                release(slot);
            };
            // Short items (the staged-epilogue instance) keep the map loop rolled, the maps'
            // statistics rotating through registers: the smaller code measured 8 % faster at
            // L = 2048, the unrolled loop 7 % faster at L = 32768.
            auto stats_tile = [&](int j, auto first, auto masked) {
                if constexpr (kStageOut) {
#pragma unroll 1
                    for (int m = 0; m < M; ++m) {
                        stats_map(j, m, mx[0], ls[0], first, masked);
                        const float m0 = mx[0], l0 = ls[0];
#pragma unroll
                        for (int q = 0; q + 1 < M; ++q) {
                            mx[q] = mx[q + 1];
                            ls[q] = ls[q + 1];
                        }
                        mx[M - 1] = m0;
                        ls[M - 1] = l0;
                    }
                } else {
                    const int k0 = j * kGBN + kq * kKQ;
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const uint32_t slot = slot_a<S>(j * M + m);
                        uint32_t x[kKQ];
                        acquire(x, slot);
                        if constexpr (decltype(masked)::value) mask_x(x, k0);
                        if constexpr (decltype(first)::value) {
                            mx[m] = fmaxf(tile_max(x), -1e30f);
                            ls[m] = tile_sum(x, mx[m]);
                        } else {
                            float ts = tile_sum(x, mx[m]);
                            if (__any_sync(0xffffffffu, !(ts <= 65536.f))) {
                                read_slot(x, slot);
                                if constexpr (decltype(masked)::value) mask_x(x, k0);
                                const float nr = fmaxf(mx[m], tile_max(x));
                                ls[m] *= fast_exp2(mx[m] - nr);
                                mx[m] = nr;
                                ts = tile_sum(x, nr);
                            }
                            ls[m] += ts;
                        }
                        release(slot);
                    }
                }
            };
            constexpr std::true_type kYes{};
            constexpr std::false_type kNo{};
            if (jfull > 0) {
                stats_tile(0, kYes, kNo);
                for (int j = 1; j < jfull; ++j) stats_tile(j, kNo, kNo);
            } else {
                stats_tile(0, kYes, kYes);
            }
            for (int j = jfull > 1 ? jfull : 1; j < it.nkv; ++j) stats_tile(j, kNo, kYes);
            // combine the four key quarters of the row: lse = max + log2(sum), base 2; the
            // exchange (P buffer 0) is written once the previous item's output stores have read
            // the P buffers
            if (kStageOut && rr > 0) {
                if (kq == 0 && lane == 0) bulk_wait_group_read<0>();
                named_bar_sync(row_bar, kRowThreads);
            }
#pragma unroll
            for (int m = 0; m < M; ++m) {
                xslot(xrow_a, kq * 8 + m) = mx[m];
                xslot(xrow_a, kq * 8 + 4 + m) = ls[m];
            }
            named_bar_sync(row_bar, kRowThreads);
            float nlse[M];                        // -lse of each map (-inf for rows past L: every P is 0)
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float mm = -INFINITY;
#pragma unroll
                for (int q = 0; q < kNQ; ++q) mm = fmaxf(mm, xslot(xrow_a, q * 8 + m));
                float lsum = 0.f;
#pragma unroll
                for (int q = 0; q < kNQ; ++q) lsum += xslot(xrow_a, q * 8 + 4 + m) * fast_exp2(xslot(xrow_a, q * 8 + m) - mm);
                nlse[m] = in ? -(mm + __log2f(lsum)) : -INFINITY;
            }
            named_bar_sync(row_bar, kRowThreads); // all have read the exchange before P overwrites it

            // ---------------------------------------------- phase B: P_h = A1_h - lambda_h A2, P_h V_h
            // one key tile: the noise map's probabilities, then each head's P tile (the per-key
            // compare only in the masked instance)
            auto diff_tile = [&](int j, auto need_mask) {
                const int k0 = j * kGBN + kq * kKQ;
                float p2[kKQ];
                {
                    uint32_t x[kKQ];
                    load_use(x, S + (j * M) % NB);
#pragma unroll
                    for (int e = 0; e < kKQ; e += 2) {
                        float y0 = __uint_as_float(x[e]), y1 = __uint_as_float(x[e + 1]);
                        ffma2(y0, y1, sl2, sl2, nlse[0], nlse[0]);
                        p2[e] = fast_exp2(y0);
                        p2[e + 1] = fast_exp2(y1);
                    }
                }
#pragma unroll
                for (int h = 0; h < S; ++h) {
                    const float nl = nlse[1 + h], nlam = -lam[h];
                    uint32_t x[kKQ];
                    load_use(x, S + (j * M + 1 + h) % NB);   // the slot is free again
                    // this thread's keys of its P half, in the K-major 128-byte-swizzled layout
                    // of the value MMA's A operand (16-byte chunk c of row t at chunk c ^ (t % 8));
                    // written once the value MMA two P tiles back has read the buffer
                    const uint32_t pb = pk & 1;
                    if (pk >= 2 && !wait_fast(&ctl->p_empty[pb][half], ((pk >> 1) - 1) & 1, p.err, abort_flag))
                        ok = false;
                    uint8_t *prow = pbuf0 + pb * 2 * LY::PH_BYTES;
#pragma unroll
                    for (int pc = 0; pc < kKQ / 32; ++pc) {
                        uint32_t pw[16];
#pragma unroll
                        for (int e2 = 0; e2 < 32; e2 += 2) {
                            const int e = pc * 32 + e2;
                            float y0 = __uint_as_float(x[e]), y1 = __uint_as_float(x[e + 1]);
                            ffma2(y0, y1, sl2, sl2, nl, nl);
                            float q0 = p2[e], q1 = p2[e + 1];
                            ffma2(q0, q1, nlam, nlam, fast_exp2(y0), fast_exp2(y1));   // P = p1 - lambda p2
                            if constexpr (decltype(need_mask)::value) {
                                if (k0 + e > last_key) q0 = 0.f;
                                if (k0 + e + 1 > last_key) q1 = 0.f;
                            }
                            pw[e2 / 2] = pack_bf16x2(q0, q1);
                        }
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int ch = chunk0 + pc * 4 + c;
                            *reinterpret_cast<uint4 *>(prow + ((ch ^ (row & 7)) << 4)) =
                                make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    lanes_arrive(&ctl->p_full[pb][half]);
                    ++pk;
                }
            };
            for (int j = 0; j < jfull; ++j) diff_tile(j, kNo);
            for (int j = jfull; j < it.nkv; ++j) diff_tile(j, kYes);

            // ---------------------------------------------- epilogue: headwise norm of each head
            ok = __all_sync(0xffffffffu, ok) && !*abort_flag;
            if (ok) ok = warp_wait_fast(&ctl->o_final, rr & 1, p.err, abort_flag);
            tc_fence_after();
            // the item's value MMAs are complete: the row's P bytes may hold the exchange again;
            // this thread's output columns of each head are [kKQ kq, kKQ kq + kKQ)
#pragma unroll
            for (int h = 0; h < S; ++h) {
                float ss = 0.f;
                if (ok) {
#pragma unroll
                    for (int c = 0; c < kKQ / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_off + 128 * h + kq * kKQ + c * 32, o);
                        tmem_ld_wait_regs(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ss = fmaf(__uint_as_float(o[e]), __uint_as_float(o[e]), ss);
                    }
                }
                xslot(xrow_b, kq * 4 + h) = ss;
            }
            named_bar_sync(row_bar, kRowThreads);
            ok = __all_sync(0xffffffffu, ok);
            if constexpr (kStageOut) {
                float yscale[S];
#pragma unroll
                for (int h = 0; h < S; ++h) {
                    float ss_tot = 0.f;
#pragma unroll
                    for (int q = 0; q < kNQ; ++q) ss_tot += xslot(xrow_b, q * 4 + h);
                    yscale[h] = p.no_norm ? 1.f : (1.f - p.lambda_init) * rsqrtf(ss_tot / 128.f + p.eps);
                }
                // The row quarter's output tile of head h is staged in P buffer 1 (h even) or 0 (h odd),
                // in the same 128-byte-swizzled halves as a P tile, and written by two TMA stores of
                // 32 rows x 64 columns issued by one thread of the quarter (rows past L are clipped).
                // Per-thread row stores would send each warp instruction to 32 different cache lines.
                named_bar_sync(row_bar, kRowThreads);   // the exchange has been read: buffer 0 is free
                const bool leader = kq == 0 && lane == 0;
                const bool rows_in = it.q0 + quarter * 32 < p.L;
                // head h's kKQ columns of this thread, normalised and packed to bf16
                auto pack = [&](int h, uint32_t (&pko)[kKQ / 2]) {
#pragma unroll
                    for (int c = 0; c < kKQ / 32; ++c) {
                        uint32_t o[32];
                        if (ok) {
                            tmem_ld32(tmem + lane_off + 128 * h + kq * kKQ + c * 32, o);
                            tmem_ld_wait_regs(o);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = 0u;
                        }
#pragma unroll
                        for (int e = 0; e < 32; e += 2)
                            pko[c * 16 + e / 2] =
                                pack_bf16x2(__uint_as_float(o[e]) * yscale[h], __uint_as_float(o[e + 1]) * yscale[h]);
                    }
                };
                auto put = [&](int h, const uint32_t (&pko)[kKQ / 2]) {
                    uint8_t *prow = pbuf0 + ((h & 1) ? 0 : 2 * LY::PH_BYTES);
#pragma unroll
                    for (int v4 = 0; v4 < kKQ / 8; ++v4)
                        *reinterpret_cast<uint4 *>(prow + (((chunk0 + v4) ^ (row & 7)) << 4)) =
                            make_uint4(pko[4 * v4], pko[4 * v4 + 1], pko[4 * v4 + 2], pko[4 * v4 + 3]);
                };
                auto store = [&](int h) {
                    if (!leader || !ok || !rows_in) return;
                    const uint8_t *src = smem + LY::OFF_P + ((h & 1) ? 0 : 2 * LY::PH_BYTES) + quarter * 32 * 128;
                    tma_store_4d(&tmO, src, 0, it.h0 + h, it.q0 + quarter * 32, it.b);
                    tma_store_4d(&tmO, src + LY::PH_BYTES, kPH, it.h0 + h, it.q0 + quarter * 32, it.b);
                    bulk_commit_group();
                };
                {
                    uint32_t pko[kKQ / 2];
                    pack(0, pko);
                    put(0, pko);
                    if constexpr (S > 1) {
                        pack(1, pko);
                        put(1, pko);
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(row_bar, kRowThreads);
                store(0);
                if constexpr (S > 1) store(1);
                uint32_t pk2[kKQ / 2];
                if constexpr (S > 2) pack(2, pk2);
                // the accumulators may now be overwritten by the next item's first value MMA
                tc_fence_before();
                lanes_arrive(&ctl->o_free);
                if constexpr (S > 2) {
                    if (leader) bulk_wait_group_read<1>();   // head 0's store has read buffer 1
                    named_bar_sync(row_bar, kRowThreads);
                    put(2, pk2);
                    fence_proxy_async_smem();
                    named_bar_sync(row_bar, kRowThreads);
                    store(2);
                }
            } else {
                // short epilogue for long items: each thread stores its own row segments
#pragma unroll
                for (int h = 0; h < S; ++h) {
                    float ss_tot = 0.f;
#pragma unroll
                    for (int q = 0; q < kNQ; ++q) ss_tot += xslot(xrow_b, q * 4 + h);
                    const float yscale =
                        p.no_norm ? 1.f : (1.f - p.lambda_init) * rsqrtf(ss_tot / 128.f + p.eps);
                    if (ok) {
#pragma unroll
                        for (int c = 0; c < kKQ / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tmem + lane_off + 128 * h + kq * kKQ + c * 32, o);
                            tmem_ld_wait_regs(o);
                            uint32_t pko[16];
#pragma unroll
                            for (int e = 0; e < 32; e += 2)
                                pko[e / 2] =
                                    pack_bf16x2(__uint_as_float(o[e]) * yscale, __uint_as_float(o[e + 1]) * yscale);
                            if (in) {
                                uint4 *dst = reinterpret_cast<uint4 *>(
                                    p.out + ((static_cast<size_t>(it.b) * p.L + qrow) * p.hs + it.h0 + h) * 128 +
                                    kq * kKQ + c * 32);
#pragma unroll
                                for (int v4 = 0; v4 < 4; ++v4)
                                    dst[v4] =
                                        make_uint4(pko[4 * v4], pko[4 * v4 + 1], pko[4 * v4 + 2], pko[4 * v4 + 3]);
                            }
                        }
                    }
                }
                // the accumulators may now be overwritten by the next item's first value MMA
                tc_fence_before();
                lanes_arrive(&ctl->o_free);
            }
            // the four warps of the row agree on whether to go on (rows share no named
            // barrier); this also orders the reads of the exchange above before the next
            // item's writes
            if (bar_red_or(row_bar, kRowThreads, !ok || *abort_flag)) break;
        }
    }

    // the store leaders (the first warp of each row quarter's column parts): stores complete
    if (kStageOut && warp >= kGCtrlWarps && warp < kGCtrlWarps + 4 && lane == 0) bulk_wait_group0();
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

template <int S, bool kStageOut>
int launch_group_impl(const PrefillArgs &a, cudaStream_t stream) {
    CUtensorMap mQ1, mK1, mQ2, mK2, mV, mO;
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
        const uint32_t box[4] = {64, 1, kPH, 1};
        if (!encode_tmap_4d_bf16(&mV, a.v, dv4, sv, box)) return GDA_ERR_CUDA;
    }
    {
        const uint64_t dout[4] = {128, hs, L, B};
        const uint64_t so[3] = {256, hs * 256, L * hs * 256};
        const uint32_t box[4] = {kPH, 1, 32, 1};
        if (!encode_tmap_4d_bf16(&mO, a.out, dout, so, box)) return GDA_ERR_CUDA;
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
    auto kern = gda_prefill_group_kernel<S, kStageOut>;
    constexpr int smem = group_smem_bytes<S>();
    static_assert(smem <= 232448, "shared memory budget");
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return record_cuda_error(e);
    // the compute warps' setmaxnreg.inc waits until the pool holds its registers: launch only
    // with the per-thread count the split was sized for
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (fa.numRegs != kGLaunchRegs) return GDA_ERR_UNSUPPORTED;
    const long long nitems = static_cast<long long>(p.nqt) * a.B * a.hn * p.nsub;
    if (nitems <= 0 || nitems > 0x7fffffffLL) return GDA_ERR_UNSUPPORTED;
    long long grid = sms;
    if (grid > nitems) grid = nitems;
    kern<<<static_cast<unsigned>(grid), kGThreads, smem, stream>>>(mQ1, mK1, mQ2, mK2, mV, mO, p);
    e = cudaGetLastError();
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

}  // namespace

bool prefill_group_supported(const PrefillArgs &a) { return a.d == 64 && a.dv == 128; }

int launch_prefill_group(const PrefillArgs &a, cudaStream_t stream) {
    if (!prefill_group_supported(a)) return GDA_ERR_UNSUPPORTED;
    int S = heads_per_item(a.hs / a.hn);
    if (S > 1) {
        // Few query tiles (a short chunk, a small batch): items of one signal head each
        // when whole groups would leave more than half of the SMs without an item.
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return record_cuda_error(e);
        const long long nqt = (a.L + kBM - 1) / kBM;
        if (2 * nqt * a.B * (a.hs / S) < sms) S = 1;
    }
    // Items of at most kStageOutTiles key tiles take the short-item instance: the staged
    // epilogue (TMA stores of the output; there the epilogue is a large share of an item) and a
    // rolled statistics loop (smaller code).  Longer items keep the per-row stores, which drain
    // while the next item's statistics sweep runs, and the unrolled loop.
    const long long Lk = a.Lk > 0 ? a.Lk : a.L;
    const bool staged = (Lk + kGBN - 1) / kGBN <= kStageOutTiles;
    switch (S) {
        case 3: return staged ? launch_group_impl<3, true>(a, stream) : launch_group_impl<3, false>(a, stream);
        case 2: return staged ? launch_group_impl<2, true>(a, stream) : launch_group_impl<2, false>(a, stream);
        default: return staged ? launch_group_impl<1, true>(a, stream) : launch_group_impl<1, false>(a, stream);
    }
}

}  // namespace gda
