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
// (h_s*dv), all bf16.  One CTA handles one (sequence, split of `chunk`
// positions) for ALL heads, so every position row is one contiguous,
// fully coalesced sweep: thread t owns the t-th 16-byte chunk of the
// concatenated [K1 | K2 | V] row and loads it with a 128-bit load for each
// position (register double buffer: the next tile's loads are in flight
// while the current tile is reduced).
//   - K threads: partial dot product over 8 dims, warp-shuffle reduction over
//     the d/8 threads of a head;
//   - one thread per head (signal and noise): online softmax in exp2 units;
//   - V threads: both accumulators O1, O2 for their 8 columns.
// Partial (m, l) per head and (O1, O2) per signal head go to the workspace;
// the combine kernel merges the splits and applies the difference and the
// (1 - lambda_init) RMSNorm epilogue.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cmath>
#include <mutex>

#include "gda.h"
#include "gda_device.cuh"
#include "gda_internal.h"

namespace gda {
namespace {

constexpr int kMaxHeads = 128;    // h_s + h_n bound for the shared score arrays

struct DecParams {
    const __nv_bfloat16 *q1, *q2, *k1c, *k2c, *vc;
    const int *lens;
    const float *lambda;
    __nv_bfloat16 *out;
    float *ws_o;       // [B][splits][hs][2][dv]
    float *ws_ml;      // [B][splits][hs+hn][2]
    unsigned *err;
    float lambda_init, eps, scale_log2;
    int B, Lcap, hs, hn, d, dv, chunk, splits;
    int kc1, kc;       // chunk boundaries: K1 chunks [0,kc1), K2 [kc1,kc), V [kc, nchunks)
    int nchunks;
};

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int clamp_len(int len, int Lcap, unsigned *err) {
    if (len < 1 || len > Lcap) {
        atomicOr(err, GDA_DEVERR_BAD_LENGTH);
        len = len < 1 ? 1 : Lcap;
    }
    return len;
}

// kTile positions per tile.  Narrow head sets (<= 384 chunks per row) run
// 4-position tiles with two CTAs per SM; wide ones 2-position tiles with up
// to 1024 threads, both without register spills.
template <int D, int kTile, int kMaxThreads, int kMinBlocks>
__global__ void __launch_bounds__(kMaxThreads, kMinBlocks)
gda_decode_split_kernel(const DecParams p) {
    // scores, then weights; double-buffered by tile parity because the K
    // threads write tile t+1's scores before the barrier that the V threads
    // of tile t pass after reading tile t's weights
    __shared__ float sc_buf[2][kMaxHeads][kTile];
    __shared__ float alpha_s[kMaxHeads];

    const int split = blockIdx.x, b = blockIdx.y;
    const int t = threadIdx.x;
    const int len = clamp_len(p.lens[b], p.Lcap, p.err);
    const int pos_begin = split * p.chunk;
    if (pos_begin >= len) return;                 // uniform over the CTA
    const int pos_end = min(len, pos_begin + p.chunk);
    const int nheads = p.hs + p.hn;
    constexpr int CPH = D / 8;                    // 16-byte chunks per head row of K

    // ---- role of this thread
    const bool is_k = t < p.kc;
    const bool is_v = t >= p.kc && t < p.nchunks;
    const size_t row_k1 = static_cast<size_t>(p.hs) * D;
    const size_t row_k2 = static_cast<size_t>(p.hn) * D;
    const size_t row_v = static_cast<size_t>(p.hs) * p.dv;
    const __nv_bfloat16 *base = nullptr;          // element address of this chunk at position 0
    size_t stride = 0;                            // elements between positions
    int sh = 0;                                   // score head of a K thread
    if (t < p.kc1) {
        base = p.k1c + static_cast<size_t>(b) * p.Lcap * row_k1 + static_cast<size_t>(t) * 8;
        stride = row_k1;
        sh = t / CPH;
    } else if (t < p.kc) {
        base = p.k2c + static_cast<size_t>(b) * p.Lcap * row_k2 + static_cast<size_t>(t - p.kc1) * 8;
        stride = row_k2;
        sh = p.hs + (t - p.kc1) / CPH;
    } else if (is_v) {
        base = p.vc + static_cast<size_t>(b) * p.Lcap * row_v + static_cast<size_t>(t - p.kc) * 8;
        stride = row_v;
    }

    // query chunk of a K thread, pre-scaled into exp2 units
    float q[8];
    if (is_k) {
        const __nv_bfloat16 *qp = (t < p.kc1)
            ? p.q1 + static_cast<size_t>(b) * row_k1 + static_cast<size_t>(t) * 8
            : p.q2 + static_cast<size_t>(b) * row_k2 + static_cast<size_t>(t - p.kc1) * 8;
        const uint4 qv = *reinterpret_cast<const uint4 *>(qp);
        const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[2 * i] = bf16_lo(w[i]) * p.scale_log2;
            q[2 * i + 1] = bf16_hi(w[i]) * p.scale_log2;
        }
    }

    // V thread: signal head and its noise head
    const int vh = is_v ? (t - p.kc) / (p.dv / 8) : 0;
    const int vg = vh / (p.hs / p.hn);
    float o1[8], o2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o1[i] = o2[i] = 0.f;
    // softmax state of head t (threads t < nheads)
    float m_run = -INFINITY, l_run = 0.f;

    auto load_tile = [&](uint4 (&buf)[kTile], int pos0) {
        if (is_k || is_v) {
#pragma unroll
            for (int i = 0; i < kTile; ++i) {
                const int pos = min(pos0 + i, pos_end - 1);   // stay inside the sequence
                buf[i] = ld_stream16(base + static_cast<size_t>(pos) * stride);
            }
        }
    };

    auto process_tile = [&](const uint4 (&buf)[kTile], int pos0, int par) {
        float (*sc)[kTile] = sc_buf[par];
        // Every lane of the warp takes part in the shuffles (a warp may hold
        // both K and V chunks); head groups of CPH lanes are CPH-aligned and
        // the K/V boundary is a multiple of CPH, so sums never mix roles.
#pragma unroll
        for (int i = 0; i < kTile; ++i) {
            float s = 0.f;
            if (is_k) {
                const uint32_t w[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s = fmaf(q[2 * e], bf16_lo(w[e]), s);
                    s = fmaf(q[2 * e + 1], bf16_hi(w[e]), s);
                }
            }
#pragma unroll
            for (int o = CPH / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (is_k && (t % CPH) == 0) sc[sh][i] = (pos0 + i < pos_end) ? s : -INFINITY;
        }
        __syncthreads();
        if (t < nheads) {
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < kTile; ++i) mt = fmaxf(mt, sc[t][i]);
            const float mn = fmaxf(m_run, mt);          // finite: position pos0 is valid
            const float a = fast_exp2(m_run - mn);      // m_run = -inf gives 0
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < kTile; ++i) {
                const float w = fast_exp2(sc[t][i] - mn);
                sc[t][i] = w;
                sum += w;
            }
            l_run = l_run * a + sum;
            m_run = mn;
            alpha_s[t] = a;
        }
        __syncthreads();
        if (is_v) {
            const float a1 = alpha_s[vh], a2 = alpha_s[p.hs + vg];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                o1[e] *= a1;
                o2[e] *= a2;
            }
#pragma unroll
            for (int i = 0; i < kTile; ++i) {
                const float w1 = sc[vh][i], w2 = sc[p.hs + vg][i];
                const uint32_t w[4] = {buf[i].x, buf[i].y, buf[i].z, buf[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float v0 = bf16_lo(w[e]), v1 = bf16_hi(w[e]);
                    o1[2 * e] = fmaf(w1, v0, o1[2 * e]);
                    o1[2 * e + 1] = fmaf(w1, v1, o1[2 * e + 1]);
                    o2[2 * e] = fmaf(w2, v0, o2[2 * e]);
                    o2[2 * e + 1] = fmaf(w2, v1, o2[2 * e + 1]);
                }
            }
        }
        // alpha_s is rewritten only after the next tile's first barrier, which
        // every V thread reaches after its reads above
    };

    const int ntiles = (pos_end - pos_begin + kTile - 1) / kTile;
    uint4 bufA[kTile], bufB[kTile];
    load_tile(bufA, pos_begin);
    for (int tile = 0; tile < ntiles; tile += 2) {
        const int pa = pos_begin + tile * kTile;
        if (tile + 1 < ntiles) load_tile(bufB, pa + kTile);
        process_tile(bufA, pa, 0);
        if (tile + 1 >= ntiles) break;
        if (tile + 2 < ntiles) load_tile(bufA, pa + 2 * kTile);
        process_tile(bufB, pa + kTile, 1);
    }

    // ---- partial state of this split
    const size_t bs = static_cast<size_t>(b) * p.splits + split;
    if (t < nheads) {
        p.ws_ml[(bs * nheads + t) * 2 + 0] = m_run;
        p.ws_ml[(bs * nheads + t) * 2 + 1] = l_run;
    }
    if (is_v) {
        const int col = (t - p.kc) % (p.dv / 8) * 8;
        float *dst = p.ws_o + ((bs * p.hs + vh) * 2) * p.dv + col;
        reinterpret_cast<float4 *>(dst)[0] = make_float4(o1[0], o1[1], o1[2], o1[3]);
        reinterpret_cast<float4 *>(dst)[1] = make_float4(o1[4], o1[5], o1[6], o1[7]);
        reinterpret_cast<float4 *>(dst + p.dv)[0] = make_float4(o2[0], o2[1], o2[2], o2[3]);
        reinterpret_cast<float4 *>(dst + p.dv)[1] = make_float4(o2[4], o2[5], o2[6], o2[7]);
    }
}

// grid (h_s, B), block dv threads: merge the splits of one (sequence, head).
__global__ void __launch_bounds__(256)
gda_decode_combine_kernel(const DecParams p) {
    __shared__ float red[8];
    const int h = blockIdx.x, b = blockIdx.y, col = threadIdx.x;
    const int g = h / (p.hs / p.hn);
    const int nheads = p.hs + p.hn;
    int len = p.lens[b];
    len = len < 1 ? 1 : (len > p.Lcap ? p.Lcap : len);
    const int ns = (len + p.chunk - 1) / p.chunk;
    const size_t b0 = static_cast<size_t>(b) * p.splits;

    float M1 = -INFINITY, M2 = -INFINITY;
    for (int s = 0; s < ns; ++s) {
        M1 = fmaxf(M1, p.ws_ml[((b0 + s) * nheads + h) * 2]);
        M2 = fmaxf(M2, p.ws_ml[((b0 + s) * nheads + p.hs + g) * 2]);
    }
    float L1 = 0.f, L2 = 0.f, O1 = 0.f, O2 = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float *ml1 = p.ws_ml + ((b0 + s) * nheads + h) * 2;
        const float *ml2 = p.ws_ml + ((b0 + s) * nheads + p.hs + g) * 2;
        const float f1 = fast_exp2(ml1[0] - M1), f2 = fast_exp2(ml2[0] - M2);
        L1 = fmaf(ml1[1], f1, L1);
        L2 = fmaf(ml2[1], f2, L2);
        const float *os = p.ws_o + (((b0 + s) * p.hs + h) * 2) * p.dv;
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

}  // namespace

DecodePlan decode_plan(int B, int Lcap, int hs, int hn, int dv) {
    DecodePlan pl;
    // 256 positions per CTA keeps >= a few waves of CTAs at serving batch
    // sizes; short caches get smaller chunks so every SM has work.
    int chunk = 256;
    while (chunk > 32 && static_cast<long long>(B) * ((Lcap + chunk - 1) / chunk) < 4 * 152) chunk /= 2;
    pl.chunk = chunk;
    pl.splits = (Lcap + chunk - 1) / chunk;
    const size_t nb = static_cast<size_t>(B) * pl.splits;
    size_t o_bytes = nb * hs * 2 * static_cast<size_t>(dv) * sizeof(float);
    o_bytes = (o_bytes + 255) / 256 * 256;
    const size_t ml_bytes = nb * (hs + hn) * 2 * sizeof(float);
    pl.bytes = o_bytes + ml_bytes;
    return pl;
}

int launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    const DecodePlan pl = decode_plan(a.B, a.Lcap, a.hs, a.hn, a.dv);
    if (a.workspace_bytes < pl.bytes) return GDA_ERR_WORKSPACE;
    DecParams p;
    p.q1 = static_cast<const __nv_bfloat16 *>(a.q1);
    p.q2 = static_cast<const __nv_bfloat16 *>(a.q2);
    p.k1c = static_cast<const __nv_bfloat16 *>(a.k1c);
    p.k2c = static_cast<const __nv_bfloat16 *>(a.k2c);
    p.vc = static_cast<const __nv_bfloat16 *>(a.vc);
    p.lens = a.lens;
    p.lambda = a.lambda;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    size_t o_bytes = static_cast<size_t>(a.B) * pl.splits * a.hs * 2 * static_cast<size_t>(a.dv) * sizeof(float);
    o_bytes = (o_bytes + 255) / 256 * 256;
    p.ws_o = static_cast<float *>(a.workspace);
    p.ws_ml = reinterpret_cast<float *>(static_cast<char *>(a.workspace) + o_bytes);
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
    p.chunk = pl.chunk;
    p.splits = pl.splits;
    p.kc1 = a.hs * a.d / 8;
    p.kc = (a.hs + a.hn) * a.d / 8;
    p.nchunks = p.kc + a.hs * a.dv / 8;
    const int threads = (p.nchunks + 31) / 32 * 32;
    if (threads > 1024 || a.hs + a.hn > kMaxHeads) return GDA_ERR_UNSUPPORTED;
    if (a.B > 65535) return GDA_ERR_UNSUPPORTED;

    dim3 grid(pl.splits, a.B);
    const bool narrow = threads <= 384;
    if (a.d == 64 && narrow)
        gda_decode_split_kernel<64, 4, 384, 2><<<grid, threads, 0, stream>>>(p);
    else if (a.d == 64)
        gda_decode_split_kernel<64, 2, 1024, 1><<<grid, threads, 0, stream>>>(p);
    else if (a.d == 128 && narrow)
        gda_decode_split_kernel<128, 4, 384, 2><<<grid, threads, 0, stream>>>(p);
    else if (a.d == 128)
        gda_decode_split_kernel<128, 2, 1024, 1><<<grid, threads, 0, stream>>>(p);
    else
        return GDA_ERR_UNSUPPORTED;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda_error(e);
    gda_decode_combine_kernel<<<dim3(a.hs, a.B), a.dv, 0, stream>>>(p);
    e = cudaGetLastError();
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
struct ScratchState {
    std::once_flag once;
    void *ptr = nullptr;
    int status = GDA_ERR_CUDA;
};
ScratchState g_scratch[kScratchDevices];

// Device address of the scratch array on the current device (set up on the
// first call for that device, with the device current).
int scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kScratchDevices) {
        cudaGetLastError();
        return GDA_ERR_CUDA;
    }
    ScratchState &s = g_scratch[dev];
    std::call_once(s.once, [&s]() {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess) {
            s.status = record_cuda_error(e);
            return;
        }
        s.ptr = ptr;
        s.status = GDA_OK;
    });
    *out = s.ptr;
    return s.status;
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

