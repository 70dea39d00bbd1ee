// Grouped differential attention decode over a bf16 KV cache (one new query
// token per sequence), split over the cache length, plus a combine pass.
//
// Operation: the last row of the causal prefill ("Differential Attention in
// Large Language Models ...", sections "Differential Attention Architecture"
// and "Headwise Normalization"; noise heads shared by groups of signal heads
// per the "Grouped Differential Attention" abstract).  The page's section
// "Hardware Implementations and Serving Considerations" places the KV cache
// on the serving path; its layout here is the plain [B, Lcap, heads, dim].
//
// Memory-bound: per cached position a sequence reads its K1 row (h_s*d),
// K2 row (h_n*d; each noise head read once for its whole group) and V row
// (h_s*dv), all bf16.  The split kernel runs two CTAs per SM (one for very
// wide rows); the batch's cache positions, concatenated sequence after
// sequence, are cut into one equal contiguous range per CTA (stream-K), so
// the load is even whatever the mix of lengths and no wave is left half
// empty.  Each CTA streams its range through a ring of shared-memory stages
// filled by 1-D bulk copies (TMA): the K1, K2 and V rows of consecutive
// positions are contiguous in the cache, so a stage is three copies issued
// by one thread, and up to 100 KB per CTA are in flight.  Every CTA handles
// ALL heads of its positions; thread t owns the t-th 16-byte chunk of the
// concatenated [K1 | K2 | V] position row and reads it from the stage:
//   - K threads: partial dot product over 8 dims, warp-shuffle reduction over
//     the d/8 threads of a head;
//   - one thread per head (signal and noise): online softmax in exp2 units;
//   - V threads: both accumulators O1, O2 for their 8 columns.
// Each (CTA, sequence) segment leaves its partial (m, l) per head and
// (O1, O2) per signal head in the workspace; the combine kernel merges a
// sequence's segments and applies the difference and the
// (1 - lambda_init) RMSNorm epilogue.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cstdint>
#include <cmath>
#include <algorithm>
#include <mutex>

#include "gda.h"
#include "gda_device.cuh"
#include "gda_internal.h"

namespace gda {
namespace {

constexpr int kMaxHeads = 128;    // h_s + h_n bound for the shared score arrays

struct DecParams {
    const __nv_bfloat16 *q1, *q2;
    const uint8_t *k1c, *k2c, *vc;    // bf16 or fp8 (e4m3) cache elements
    const float *k1_scale, *k2_scale, *v_scale;   // per-head dequantisation scales (fp8 caches)
    const int *lens;
    const float *lambda;
    __nv_bfloat16 *out;
    float *ws_o;       // [slots][hs][2][dv]     slot = CTA + sequence
    float *ws_ml;      // [slots][hs+hn][2]
    int *ws_seg;       // [B][2]: first and last CTA holding a segment of the sequence
    unsigned *err;
    float lambda_init, eps, scale_log2;
    int B, Lcap, hs, hn, d, dv;
    int min_per_cta;   // fewest positions a CTA takes
    int ctas;          // CTAs of the split kernel
    int kc1, kc;       // chunk boundaries: K1 chunks [0,kc1), K2 [kc1,kc), V [kc, nchunks)
    int nchunks;
    int es;            // cache element bytes: 2 (bf16) or 1 (fp8 e4m3)
    // paged caches: the caches are page pools [num_pages, page_size, heads,
    // dim]; position j of sequence b is row j % page_size of page
    // block_table[b * max_pages + j / page_size]
    const int *block_table;   // nullptr: contiguous caches [B, Lcap, heads, dim]
    int page_size, max_pages, num_pages;
};

__device__ __forceinline__ int clamp_len(int len, int Lcap, unsigned *err) {
    if (len < 1 || len > Lcap) {
        atomicOr(err, GDA_DEVERR_BAD_LENGTH);
        len = len < 1 ? 1 : Lcap;
    }
    return len;
}

constexpr int kMaxStages = 8;

// 1-D bulk copy (TMA) of `bytes` contiguous bytes into shared memory,
// completing on `bar` as transaction bytes.  Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ long long warp_incl_scan(long long x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Producer state (thread 0 of a CTA): a cursor over the CTA's range
// [start, end) of the batch's concatenated cache positions.  b is the
// current sequence, whose positions begin at `pre` in the concatenation;
// pos is its next position and hi the end of its part of the range.
struct Cursor {
    long long pre, end, per;
    int b, len, pos, hi, k;   // k: tiles issued so far
    int cta;
    bool done;
};

// What the consumers of a stage need to know about its tile.
struct TileInfo {
    int n;      // positions in the tile (1..P)
    int b;      // sequence
    int flags;  // kSegEnd: last tile of the CTA's segment of sequence b; kLast: last tile of the CTA
};
constexpr int kSegEnd = 1, kLast = 2;

// A segment that starts at position 0 of sequence c.b records the first and
// last CTA whose range meets the sequence (the combine kernel reads them).
__device__ __forceinline__ void note_first_segment(const DecParams &p, const Cursor &c) {
    if (c.pos != 0) return;
    p.ws_seg[2 * c.b] = c.cta;
    p.ws_seg[2 * c.b + 1] = static_cast<int>((c.pre + c.len - 1) / c.per);
}

// Issues the next tile of cursor c (if any) into stage c.k % stages: its
// TileInfo, then the three bulk copies on the stage's barrier.
template <int P>
__device__ __forceinline__ void issue_tile(const DecParams &p, Cursor &c, int stages, uint8_t *ring,
                                           uint64_t *full, TileInfo *info) {
    if (c.done) return;
    const uint32_t rk1 = p.hs * p.d * p.es, rk2 = p.hn * p.d * p.es, rv = p.hs * p.dv * p.es;
    const int n = min(P, c.hi - c.pos);
    const int st = c.k % stages;
    uint8_t *sb = ring + static_cast<size_t>(st) * P * (rk1 + rk2 + rv);
    const size_t row0 = static_cast<size_t>(c.b) * p.Lcap + c.pos;
    const int b = c.b, pos0 = c.pos;

    // advance the cursor
    int flags = 0;
    c.pos += n;
    if (c.pos >= c.hi) {
        flags = kSegEnd;
        if (c.pre + c.hi >= c.end) {
            c.done = true;
            flags |= kLast;
        } else {
            c.pre += c.len;
            ++c.b;
            c.len = clamp_len(p.lens[c.b], p.Lcap, p.err);
            c.pos = 0;
            c.hi = static_cast<int>(min(static_cast<long long>(c.len), c.end - c.pre));
            note_first_segment(p, c);
        }
    }
    info[st] = TileInfo{n, b, flags};
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // prior generic reads of the stage
    mbar_arrive_expect_tx(&full[st], n * (rk1 + rk2 + rv));          // releases info[st]
    if (p.block_table == nullptr) {
        bulk_copy_g2s(sb, p.k1c + row0 * rk1, n * rk1, &full[st]);
        bulk_copy_g2s(sb + P * rk1, p.k2c + row0 * rk2, n * rk2, &full[st]);
        bulk_copy_g2s(sb + P * (rk1 + rk2), p.vc + row0 * rv, n * rv, &full[st]);
    } else {
        // one run of rows per page the tile touches; a page id outside the
        // pool is reported and read as page 0 instead
        for (int i = 0; i < n;) {
            const int pos = pos0 + i;
            const int pg = pos / p.page_size, in_pg = pos % p.page_size;
            const int run = min(n - i, p.page_size - in_pg);
            int phys = p.block_table[static_cast<size_t>(b) * p.max_pages + pg];
            if (phys < 0 || phys >= p.num_pages) {
                atomicOr(p.err, GDA_DEVERR_BAD_PAGE);
                phys = 0;
            }
            const size_t r0 = static_cast<size_t>(phys) * p.page_size + in_pg;
            bulk_copy_g2s(sb + i * rk1, p.k1c + r0 * rk1, run * rk1, &full[st]);
            bulk_copy_g2s(sb + P * rk1 + i * rk2, p.k2c + r0 * rk2, run * rk2, &full[st]);
            bulk_copy_g2s(sb + P * (rk1 + rk2) + i * rv, p.vc + r0 * rv, run * rv, &full[st]);
            i += run;
        }
    }
    ++c.k;
}

// The EPC cache elements of one 16-byte chunk as floats: 8 bf16, or 16 fp8
// (e4m3) through the packed fp8x2 -> half2 conversion.
template <bool F8>
__device__ __forceinline__ void unpack_chunk(const uint4 &c, float (&x)[F8 ? 16 : 8]) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    if constexpr (F8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
                    static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * hh)) & 0xFFFFu), __NV_E4M3);
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
                x[4 * i + 2 * hh] = f.x;
                x[4 * i + 2 * hh + 1] = f.y;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = bf16_lo(w[i]);
            x[2 * i + 1] = bf16_hi(w[i]);
        }
    }
}

// P consecutive floats from shared memory (16-byte aligned for P >= 4, 8-byte for P = 2).
template <int P>
__device__ __forceinline__ void load_weights(float (&w)[P], const float *src) {
    if constexpr (P % 4 == 0) {
#pragma unroll
        for (int i = 0; i < P; i += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src + i);
            w[i] = x.x;
            w[i + 1] = x.y;
            w[i + 2] = x.z;
            w[i + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < P; i += 2) {
            const float2 x = *reinterpret_cast<const float2 *>(src + i);
            w[i] = x.x;
            w[i + 1] = x.y;
        }
    }
}

// Stream-K split of the cache: the batch's cache positions, concatenated
// sequence after sequence, are cut into gridDim.x equal contiguous ranges,
// one per CTA, so every CTA streams the same number of bytes whatever the
// mix of lengths.  A range may span several sequences; the part of it in
// one sequence is a segment, and each segment leaves one partial softmax
// state in workspace slot (CTA + sequence) (unique: along the position axis
// neither index decreases and at least one grows at each segment change).
//
// Warp roles, decoupled by mbarriers (no CTA-wide barrier per tile):
//   - warp 0, one thread: producer.  Streams the range through a ring of
//     `stages` shared-memory stages of P positions: per stage its TileInfo
//     and three bulk copies (the K1, K2 and V rows of P consecutive
//     positions of one sequence, contiguous in the cache).  Positions
//     outside the range are never copied.
//   - K warps: thread (32 + c) owns the c-th 16-byte chunk of the
//     concatenated [K1 | K2] row: 8-dim partial dot products, reduced over
//     the head's d/8 lanes by shuffles, after which every lane of the head
//     holds the head's P scores and runs the head's online softmax
//     (exp2 units) redundantly; the head's weights and rescale factor go to
//     the stage's weight slot, then the warp arrives on wready[stage].
//   - V warps (from the next warp boundary): one 16-byte chunk of the V row
//     each; wait for wready, rescale and accumulate O1 (signal weights) and
//     O2 (weights of the head's noise head) for 8 columns, arrive on
//     empty[stage], which hands the stage back to the producer.
// Shared memory (dynamic): ring [stages][P rows of K1 | P rows of K2 |
// P rows of V], weights [stages][h_s + h_n][P], rescale [stages][h_s + h_n].
template <int D, int P, bool F8, int kMaxThreads, int kMinBlocks>
__global__ void __launch_bounds__(kMaxThreads, kMinBlocks)
gda_decode_split_kernel(const DecParams p, int stages) {
    constexpr int EPC = F8 ? 16 : 8;              // cache elements per 16-byte chunk
    __shared__ uint64_t full[kMaxStages], wready[kMaxStages], empty[kMaxStages];
    __shared__ TileInfo info[kMaxStages];
    __shared__ long long red_s[32];
    __shared__ long long found_pre;
    __shared__ int found_b;
    __shared__ int abort_flag;
    extern __shared__ __align__(128) uint8_t ring[];

    const int cta = blockIdx.x;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = blockDim.x >> 5;

    // ---- total positions of the batch, and this CTA's range
    long long part = 0;
    for (int b = t; b < p.B; b += blockDim.x) part += clamp_len(p.lens[b], p.Lcap, p.err);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red_s[warp] = part;
    if (t == 0) found_b = -1;
    __syncthreads();
    long long total = 0;
    for (int w = 0; w < nwarps; ++w) total += red_s[w];
    long long per = (total + gridDim.x - 1) / gridDim.x;
    if (per < p.min_per_cta) per = p.min_per_cta;
    const long long start = static_cast<long long>(cta) * per;
    if (start >= total) return;                   // uniform over the CTA

    // ---- the sequence holding position `start`: block-wide scan of the lengths
    long long carry = 0;
    for (int base = 0; base < p.B; base += blockDim.x) {
        __syncthreads();                           // red_s reads of the previous pass are done
        const int b = base + t;
        const long long len = b < p.B ? clamp_len(p.lens[b], p.Lcap, p.err) : 0;
        const long long incl = warp_incl_scan(len);
        if (lane == 31) red_s[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            long long w = lane < nwarps ? red_s[lane] : 0;
            w = warp_incl_scan(w);
            if (lane < nwarps) red_s[lane] = w;
        }
        __syncthreads();
        const long long before = carry + (warp > 0 ? red_s[warp - 1] : 0) + incl - len;
        if (b < p.B && before <= start && start < before + len) {
            found_b = b;
            found_pre = before;
        }
        carry += red_s[nwarps - 1];
        __syncthreads();
        if (found_b >= 0) break;                   // uniform
    }
    if (found_b < 0) return;                       // unreachable while every length is >= 1

    const int nheads = p.hs + p.hn;
    const int n_kwarps = (p.kc + 31) / 32;
    const int vbase = 32 + n_kwarps * 32;          // first V thread
    const int n_vwarps = (p.nchunks - p.kc + 31) / 32;
    const uint32_t rk1 = p.hs * D * p.es, rk2 = p.hn * D * p.es, rv = p.hs * p.dv * p.es;   // row bytes
    const uint32_t stage_bytes = P * (rk1 + rk2 + rv);
    float *wts = reinterpret_cast<float *>(ring + static_cast<size_t>(stages) * stage_bytes);  // [stages][nheads][P]
    float *alph = wts + stages * nheads * P;                                                    // [stages][nheads]

    if (t == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&wready[s], n_kwarps);
            mbar_init(&empty[s], n_vwarps);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    const int b_first = found_b;
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
        Cursor c;
        c.pre = found_pre;
        c.end = min(total, start + per);
        c.per = per;
        c.b = b_first;
        c.len = clamp_len(p.lens[c.b], p.Lcap, p.err);
        c.pos = static_cast<int>(start - c.pre);
        c.hi = static_cast<int>(min(static_cast<long long>(c.len), c.end - c.pre));
        c.k = 0;
        c.cta = cta;
        c.done = false;
        note_first_segment(p, c);
        while (!c.done) {
            if (c.k >= stages &&
                !mbar_wait(&empty[c.k % stages], ((c.k / stages) - 1) & 1, p.err, GDA_DEVERR_DECODE_TIMEOUT,
                           &abort_flag))
                return;
            issue_tile<P>(p, c, stages, ring, full, info);
        }
        return;
    }

    if (t < vbase) {
        // ------------------------------------------------------ K warps
        constexpr int CPH = D / EPC;               // lanes (16-byte chunks) per head row of K
        const int kk = t - 32;                     // chunk index in [K1 | K2]
        const bool is_k = kk < p.kc;
        uint32_t off = 0, stride = 0;
        int sh = 0;                                // score head
        if (kk < p.kc1) {
            off = kk * 16;
            stride = rk1;
            sh = kk / CPH;
        } else if (is_k) {
            off = P * rk1 + (kk - p.kc1) * 16;
            stride = rk2;
            sh = p.hs + (kk - p.kc1) / CPH;
        }
        const int gl = kk % CPH;                   // lane within the head's group

        // query chunk of a K thread, pre-scaled into exp2 units (and by the
        // head's K dequantisation scale for an fp8 cache)
        float q[EPC];
        auto load_q = [&](int b) {
#pragma unroll
            for (int i = 0; i < EPC; ++i) q[i] = 0.f;
            if (!is_k) return;
            const bool sig = kk < p.kc1;
            const int c = sig ? kk : kk - p.kc1;
            const __nv_bfloat16 *qp = sig ? p.q1 + static_cast<size_t>(b) * p.hs * D + static_cast<size_t>(c) * EPC
                                          : p.q2 + static_cast<size_t>(b) * p.hn * D + static_cast<size_t>(c) * EPC;
            float f = p.scale_log2;
            if constexpr (F8) f *= sig ? p.k1_scale[sh] : p.k2_scale[sh - p.hs];
#pragma unroll
            for (int h8 = 0; h8 < EPC / 8; ++h8) {
                const uint4 qv = reinterpret_cast<const uint4 *>(qp)[h8];
                const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    q[8 * h8 + 2 * i] = bf16_lo(w[i]) * f;
                    q[8 * h8 + 2 * i + 1] = bf16_hi(w[i]) * f;
                }
            }
        };
        load_q(b_first);
        float m_run = -INFINITY, l_run = 0.f;     // softmax state of head sh

        for (int it = 0;; ++it) {
            const int st = it % stages;
            // warp-uniform outcome: the shuffles below need every lane
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&full[st], (it / stages) & 1, p.err, GDA_DEVERR_DECODE_TIMEOUT, &abort_flag)))
                return;
            const TileInfo ti = info[st];
            const uint8_t *sb = ring + static_cast<size_t>(st) * stage_bytes + off;
            float s[P];
#pragma unroll
            for (int i = 0; i < P; ++i) {
                float a0 = 0.f, a1 = 0.f;
                if (is_k && i < ti.n) {
                    float kx[EPC];
                    unpack_chunk<F8>(*reinterpret_cast<const uint4 *>(sb + i * stride), kx);
#pragma unroll
                    for (int e = 0; e < EPC; e += 2) ffma2_acc(a0, a1, q[e], q[e + 1], kx[e], kx[e + 1]);
                }
                s[i] = a0 + a1;
            }
            // head sums over the CPH lanes of each head (CPH-aligned groups;
            // lanes past the K chunks hold zeros and form their own groups)
#pragma unroll
            for (int o = CPH / 2; o > 0; o >>= 1)
#pragma unroll
                for (int i = 0; i < P; ++i) s[i] += __shfl_xor_sync(0xffffffffu, s[i], o);
            // online softmax of head sh, identical on every lane of the group
            float mt = m_run;
#pragma unroll
            for (int i = 0; i < P; ++i) {
                if (i >= ti.n) s[i] = -INFINITY;
                mt = fmaxf(mt, s[i]);
            }
            const float a = fast_exp2(m_run - mt);    // m_run = -inf gives 0
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < P; ++i) {
                s[i] = fast_exp2(s[i] - mt);
                sum += s[i];
            }
            l_run = l_run * a + sum;
            m_run = mt;
            if (is_k) {
                float *wrow = wts + (st * nheads + sh) * P;
                // every lane of the group holds all P weights; lane gl writes
                // the positions i with i % CPH == gl (CPH may be below P)
#pragma unroll
                for (int i = 0; i < P; ++i)
                    if (gl == i % CPH) wrow[i] = s[i];
                if (gl == 0) alph[st * nheads + sh] = a;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&wready[st]);

            if (ti.flags & kSegEnd) {
                if (is_k && gl == 0) {
                    const size_t slot = static_cast<size_t>(cta) + ti.b;
                    p.ws_ml[(slot * nheads + sh) * 2 + 0] = m_run;
                    p.ws_ml[(slot * nheads + sh) * 2 + 1] = l_run;
                }
                if (ti.flags & kLast) return;
                m_run = -INFINITY;
                l_run = 0.f;
                load_q(ti.b + 1);                      // segments follow the sequences in order
            }
        }
    }

    // ---------------------------------------------------------- V warps
    const int vv = t - vbase;                      // chunk index in the V row
    const bool is_v = vv < p.hs * p.dv / EPC;
    const int vh = is_v ? vv / (p.dv / EPC) : 0;   // signal head
    const int vg = p.hs + vh / (p.hs / p.hn);      // its noise head's score index
    const int vcol = is_v ? vv % (p.dv / EPC) * EPC : 0;
    const uint32_t off = P * (rk1 + rk2) + (is_v ? vv : 0) * 16;
    float o1[EPC], o2[EPC];
#pragma unroll
    for (int i = 0; i < EPC; ++i) o1[i] = o2[i] = 0.f;

    for (int it = 0;; ++it) {
        const int st = it % stages;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&wready[st], (it / stages) & 1, p.err, GDA_DEVERR_DECODE_TIMEOUT, &abort_flag)))
            return;
        const TileInfo ti = info[st];
        if (is_v) {
            const float a1 = alph[st * nheads + vh], a2 = alph[st * nheads + vg];
            float w1[P], w2[P];
            load_weights<P>(w1, wts + (st * nheads + vh) * P);
            load_weights<P>(w2, wts + (st * nheads + vg) * P);
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                o1[e] *= a1;
                o2[e] *= a2;
            }
            const uint8_t *sb = ring + static_cast<size_t>(st) * stage_bytes + off;
#pragma unroll
            for (int i = 0; i < P; ++i) {
                if (i >= ti.n) break;                  // rows outside the range were never copied
                float vx[EPC];
                unpack_chunk<F8>(*reinterpret_cast<const uint4 *>(sb + i * rv), vx);
#pragma unroll
                for (int e = 0; e < EPC; e += 2) {
                    ffma2_acc(o1[e], o1[e + 1], w1[i], w1[i], vx[e], vx[e + 1]);
                    ffma2_acc(o2[e], o2[e + 1], w2[i], w2[i], vx[e], vx[e + 1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);

        if (ti.flags & kSegEnd) {
            // end of a segment: its partial state goes to slot (CTA + sequence)
            if (is_v) {
                const size_t slot = static_cast<size_t>(cta) + ti.b;
                float *dst = p.ws_o + ((slot * p.hs + vh) * 2) * p.dv + vcol;
                // an fp8 cache's V scale multiplies the whole accumulator
                const float vs = F8 ? p.v_scale[vh] : 1.f;
#pragma unroll
                for (int e = 0; e < EPC; e += 4) {
                    reinterpret_cast<float4 *>(dst)[e / 4] =
                        make_float4(o1[e] * vs, o1[e + 1] * vs, o1[e + 2] * vs, o1[e + 3] * vs);
                    reinterpret_cast<float4 *>(dst + p.dv)[e / 4] =
                        make_float4(o2[e] * vs, o2[e + 1] * vs, o2[e + 2] * vs, o2[e + 3] * vs);
                }
            }
            if (ti.flags & kLast) return;
#pragma unroll
            for (int i = 0; i < EPC; ++i) o1[i] = o2[i] = 0.f;
        }
    }
}

// grid (h_s, B), block dv threads: merge the segments of one (sequence, head).
__global__ void __launch_bounds__(256)
gda_decode_combine_kernel(const DecParams p) {
    // launched as a programmatic dependent of the split kernel: its launch overlaps the split
    // kernel's tail, and this wait returns once that grid has completed with its writes visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float red[8];
    const int h = blockIdx.x, b = blockIdx.y, col = threadIdx.x;
    const int g = h / (p.hs / p.hn);
    const int nheads = p.hs + p.hn;
    // CTAs c0..c1 left a segment of this sequence in slots c + b (clamped so
    // that a damaged workspace cannot send the reads out of bounds)
    const int c0 = min(max(p.ws_seg[2 * b], 0), p.ctas - 1);
    const int c1 = min(max(p.ws_seg[2 * b + 1], c0), p.ctas - 1);

    float M1 = -INFINITY, M2 = -INFINITY;
    for (int c = c0; c <= c1; ++c) {
        const size_t slot = static_cast<size_t>(c) + b;
        M1 = fmaxf(M1, p.ws_ml[(slot * nheads + h) * 2]);
        M2 = fmaxf(M2, p.ws_ml[(slot * nheads + p.hs + g) * 2]);
    }
    float L1 = 0.f, L2 = 0.f, O1 = 0.f, O2 = 0.f;
    for (int c = c0; c <= c1; ++c) {
        const size_t slot = static_cast<size_t>(c) + b;
        const float *ml1 = p.ws_ml + (slot * nheads + h) * 2;
        const float *ml2 = p.ws_ml + (slot * nheads + p.hs + g) * 2;
        const float f1 = fast_exp2(ml1[0] - M1), f2 = fast_exp2(ml2[0] - M2);
        L1 = fmaf(ml1[1], f1, L1);
        L2 = fmaf(ml2[1], f2, L2);
        const float *os = p.ws_o + ((slot * p.hs + h) * 2) * p.dv;
        O1 = fmaf(os[col], f1, O1);
        O2 = fmaf(os[p.dv + col], f2, O2);
    }
    const float o = O1 / L1 - p.lambda[h] * (O2 / L2);
    float ss = o * o;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((col & 31) == 0) red[col >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (p.dv + 31) / 32; ++w) tot += red[w];
    const float y = (1.f - p.lambda_init) * o * rsqrtf(tot / static_cast<float>(p.dv) + p.eps);
    p.out[(static_cast<size_t>(b) * p.hs + h) * p.dv + col] = __float2bfloat16_rn(y);
}

template <int D, int P, bool F8>
cudaError_t launch_split(dim3 grid, int threads, size_t smem, cudaStream_t stream, const DecParams &p, int stages) {
    // up to 256 threads: three CTAs per SM with up to 85 registers a thread;
    // up to 384: two with up to 80; else at most 64 registers (two CTAs of
    // up to 512 threads, or one)
    auto kern = threads <= 256   ? gda_decode_split_kernel<D, P, F8, 256, 3>
                : threads <= 384 ? gda_decode_split_kernel<D, P, F8, 384, 2>
                                 : gda_decode_split_kernel<D, P, F8, 1024, 1>;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, threads, smem, stream>>>(p, stages);
    return cudaSuccess;
}

}  // namespace

// Upper bound on the split kernel's CTAs (four per SM on a 152-SM part); the
// workspace holds one partial state per (CTA + sequence) slot.
constexpr int kDecodeMaxCtas = 608;

DecodePlan decode_plan(int B, int Lcap, int hs, int hn, int dv) {
    (void)Lcap;
    DecodePlan pl;
    pl.slots = kDecodeMaxCtas + B;
    pl.o_bytes = (static_cast<size_t>(pl.slots) * hs * 2 * dv * sizeof(float) + 255) / 256 * 256;
    pl.ml_bytes = (static_cast<size_t>(pl.slots) * (hs + hn) * 2 * sizeof(float) + 255) / 256 * 256;
    pl.bytes = pl.o_bytes + pl.ml_bytes + static_cast<size_t>(B) * 2 * sizeof(int);
    return pl;
}

int launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    const DecodePlan pl = decode_plan(a.B, a.Lcap, a.hs, a.hn, a.dv);
    if (a.workspace_bytes < pl.bytes) return GDA_ERR_WORKSPACE;
    DecParams p;
    p.q1 = static_cast<const __nv_bfloat16 *>(a.q1);
    p.q2 = static_cast<const __nv_bfloat16 *>(a.q2);
    p.k1c = static_cast<const uint8_t *>(a.k1c);
    p.k2c = static_cast<const uint8_t *>(a.k2c);
    p.vc = static_cast<const uint8_t *>(a.vc);
    p.block_table = a.block_table;
    p.page_size = a.page_size;
    p.max_pages = a.max_pages;
    p.num_pages = a.num_pages;
    p.k1_scale = a.k1_scale;
    p.k2_scale = a.k2_scale;
    p.v_scale = a.v_scale;
    const bool f8 = a.fp8 != 0;
    const int epc = f8 ? 16 : 8;                  // cache elements per 16-byte chunk
    p.es = f8 ? 1 : 2;
    p.lens = a.lens;
    p.lambda = a.lambda;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.ws_o = static_cast<float *>(a.workspace);
    p.ws_ml = reinterpret_cast<float *>(static_cast<char *>(a.workspace) + pl.o_bytes);
    p.ws_seg = reinterpret_cast<int *>(static_cast<char *>(a.workspace) + pl.o_bytes + pl.ml_bytes);
    p.err = a.dev_err;
    p.lambda_init = a.lambda_init;
    p.eps = a.eps;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.d)));
    p.B = a.B;
    p.Lcap = a.Lcap;
    p.hs = a.hs;
    p.hn = a.hn;
    p.d = a.d;
    p.dv = a.dv;
    p.kc1 = a.hs * a.d / epc;
    p.kc = (a.hs + a.hn) * a.d / epc;
    p.nchunks = p.kc + a.hs * a.dv / epc;
    // producer warp, K warps, V warps (each role starts on a warp boundary)
    const int threads = 32 + (p.kc + 31) / 32 * 32 + (p.nchunks - p.kc + 31) / 32 * 32;
    if (threads > 1024 || a.hs + a.hn > kMaxHeads) return GDA_ERR_UNSUPPORTED;
    if (a.B > 65535) return GDA_ERR_UNSUPPORTED;

    // every copy in flight completes within the CTA's range (no position
    // outside it is copied), so the CTA can exit after its last tile
    const size_t row_bytes = p.es * (static_cast<size_t>(a.hs) * a.d + static_cast<size_t>(a.hn) * a.d +
                                     static_cast<size_t>(a.hs) * a.dv);
    const int nheads = a.hs + a.hn;
    // ring budget: four CTAs per SM for an fp8 cache whose CTA has at most
    // 192 threads (measured 4.74 against 4.48 TB/s with three CTAs of three
    // stages: the widening and multiply-adds need the extra warps), three
    // when a CTA has at most 256 threads, two up to 512, else one (each with
    // its static arrays within 228 KB); the largest stage of 8, 4 or 2
    // positions of which at least the minimum count fits (a stage also holds
    // its P weights and rescale factor per head)
    const int per_sm = (f8 && threads <= 192) ? 4 : (threads <= 256 ? 3 : (threads <= 512 ? 2 : 1));
    const size_t budget =
        per_sm == 4 ? 52 * 1024 : (per_sm == 3 ? 70 * 1024 : (per_sm == 2 ? 100 * 1024 : 200 * 1024));
    int P = 8;
    const size_t min_stages = per_sm == 4 ? 2 : (per_sm == 3 ? 3 : 4);
    while (P > 2 && (row_bytes * P + nheads * (P + 1) * 4) * min_stages > budget) P /= 2;
    const size_t per_stage = row_bytes * P + static_cast<size_t>(nheads) * (P + 1) * 4;
    int stages = static_cast<int>(budget / per_stage);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return GDA_ERR_UNSUPPORTED;
    const size_t smem = static_cast<size_t>(stages) * per_stage;
    int dev = 0, sms = 0;
    cudaError_t e1 = cudaGetDevice(&dev);
    if (e1 == cudaSuccess) e1 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e1 != cudaSuccess) return record_cuda_error(e1);
    p.ctas = std::min(kDecodeMaxCtas, per_sm * sms);
    p.min_per_cta = 64;
    const dim3 grid(p.ctas);
    cudaError_t e0;
    switch ((a.d * 16 + P) * 2 + (f8 ? 1 : 0)) {
        case (64 * 16 + 8) * 2: e0 = launch_split<64, 8, false>(grid, threads, smem, stream, p, stages); break;
        case (64 * 16 + 4) * 2: e0 = launch_split<64, 4, false>(grid, threads, smem, stream, p, stages); break;
        case (64 * 16 + 2) * 2: e0 = launch_split<64, 2, false>(grid, threads, smem, stream, p, stages); break;
        case (128 * 16 + 8) * 2: e0 = launch_split<128, 8, false>(grid, threads, smem, stream, p, stages); break;
        case (128 * 16 + 4) * 2: e0 = launch_split<128, 4, false>(grid, threads, smem, stream, p, stages); break;
        case (128 * 16 + 2) * 2: e0 = launch_split<128, 2, false>(grid, threads, smem, stream, p, stages); break;
        case (64 * 16 + 8) * 2 + 1: e0 = launch_split<64, 8, true>(grid, threads, smem, stream, p, stages); break;
        case (64 * 16 + 4) * 2 + 1: e0 = launch_split<64, 4, true>(grid, threads, smem, stream, p, stages); break;
        case (128 * 16 + 8) * 2 + 1: e0 = launch_split<128, 8, true>(grid, threads, smem, stream, p, stages); break;
        case (128 * 16 + 4) * 2 + 1: e0 = launch_split<128, 4, true>(grid, threads, smem, stream, p, stages); break;
        case (64 * 16 + 2) * 2 + 1: e0 = launch_split<64, 2, true>(grid, threads, smem, stream, p, stages); break;
        case (128 * 16 + 2) * 2 + 1: e0 = launch_split<128, 2, true>(grid, threads, smem, stream, p, stages); break;
        default: return GDA_ERR_UNSUPPORTED;
    }
    if (e0 != cudaSuccess) return record_cuda_error(e0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda_error(e);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.hs, a.B);
    cfg.blockDim = dim3(a.dv);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gda_decode_combine_kernel, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

}  // namespace gda

// ------------------------------------------------------------------------
// Decode without any device allocation.
//
// Some callers cannot hand this library a workspace: for instance a plugin
// or serving loop that owns no allocator (the host framework holds all
// device memory in its own pool), or code that must never call cudaMalloc /
// cudaFree because those calls can synchronise the device and stall other
// work.  For them the decode's split partials live in one fixed scratch
// array that is part of the library itself.  The array is a file-scope
// __device__ object: every device that loads the library keeps its
// GDA_DECODE_SCRATCH_BYTES until the process exits.  Host code may not use
// the array's name as a pointer (on the host it is only a stand-in), so the
// device address is fetched once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[GDA_DECODE_SCRATCH_BYTES];

namespace gda {
namespace {
constexpr int kScratchDevices = 64;
// Per device: the scratch array's device address once a lookup succeeded.
// A failed lookup (for instance one made during a stream capture) is not
// remembered, so a later call on that device tries again.
struct ScratchState {
    std::mutex mu;
    void *ptr = nullptr;
};
ScratchState g_scratch[kScratchDevices];

// Device address of the scratch array on the current device (looked up with
// the device current, on the first successful call for that device).
int scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kScratchDevices) {
        cudaGetLastError();
        return GDA_ERR_CUDA;
    }
    ScratchState &s = g_scratch[dev];
    std::lock_guard<std::mutex> lock(s.mu);
    if (s.ptr == nullptr) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess) return record_cuda_error(e);
        s.ptr = ptr;
    }
    *out = s.ptr;
    return GDA_OK;
}
}  // namespace

}  // namespace gda

extern "C" int gda_attn_decode_noalloc(const void *q_sig, const void *q_noise, const void *k_sig_cache,
                                       const void *k_noise_cache, const void *v_cache,
                                       const int *cache_lens, const float *lambda, float lambda_init,
                                       void *out, int B, int Lcap, int h_s, int h_n, int d, int dv,
                                       float eps, gda_stream_t stream) {
    const size_t need = gda_attn_decode_workspace_size(B, Lcap, h_s, h_n, dv);
    if (need > static_cast<size_t>(GDA_DECODE_SCRATCH_BYTES)) return GDA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        const int st = gda::scratch_address(&scratch);
        if (st != GDA_OK) return st;
    }
    // invalid sizes (need == 0) are reported by the regular entry point
    return gda_attn_decode(q_sig, q_noise, k_sig_cache, k_noise_cache, v_cache, cache_lens, lambda,
                           lambda_init, out, B, Lcap, h_s, h_n, d, dv, eps, scratch,
                           static_cast<size_t>(GDA_DECODE_SCRATCH_BYTES), stream);
}

