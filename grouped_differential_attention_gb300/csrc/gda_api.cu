// C ABI of libgda.so (declared in include/gda.h): argument validation,
// device checks, TMA descriptor encoding and dispatch to the kernels.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "gda.h"
#include "gda_internal.h"

// Device error word (one per device that loads the library).  Kernels set
// GDA_DEVERR_* bits here instead of trapping.
__device__ unsigned g_gda_device_error;

namespace gda {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::once_flag once;
    int status = GDA_ERR_CUDA;     // GDA_OK once the device checked out
    unsigned *err_word = nullptr;  // device address of g_gda_device_error
};
DeviceState g_dev[kMaxDevices];

// Checks the current device once: compute capability 10.3 (GB300) and the
// address of the error word.  Returns a gda_status and the word's address.
int current_device(unsigned **err_word) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GDA_ERR_CUDA;
    }
    DeviceState &s = g_dev[dev];
    std::call_once(s.once, [&s, dev]() {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            s.status = GDA_ERR_CUDA;
            return;
        }
        if (major != 10 || minor != 3) {
            s.status = GDA_ERR_UNSUPPORTED;
            return;
        }
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_gda_device_error) != cudaSuccess) {
            cudaGetLastError();
            s.status = GDA_ERR_CUDA;
            return;
        }
        s.err_word = static_cast<unsigned *>(addr);
        s.status = GDA_OK;
    });
    *err_word = s.err_word;
    return s.status;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_prefill_common(const void *q1, const void *k1, const void *q2, const void *k2,
                         const void *v, const float *lam, float lambda_init, const void *out, int B,
                         int L, int hs, int hn, int d, int dv, int causal, float eps,
                         unsigned flags, unsigned allowed_flags = GDA_FLAG_NO_NORM) {
    if (!q1 || !k1 || !q2 || !k2 || !v || !lam || !out) return GDA_ERR_INVALID_ARG;
    if (B < 1 || L < 1 || hs < 1 || hn < 1 || d < 1 || dv < 1) return GDA_ERR_INVALID_ARG;
    if (hs % hn != 0) return GDA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return GDA_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(lambda_init)) return GDA_ERR_INVALID_ARG;
    if (flags & ~allowed_flags) return GDA_ERR_INVALID_ARG;
    // element counts must fit the 64-bit index arithmetic with room to spare
    const double elems = static_cast<double>(B) * L * (hs > hn ? hs : hn) * (d > dv ? d : dv);
    if (elems > 9.0e15) return GDA_ERR_INVALID_ARG;
    if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
        !aligned16(lam) || !aligned16(out))
        return GDA_ERR_MISALIGNED;
    return GDA_OK;
}

thread_local int g_last_cuda_error = 0;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

int device_state(unsigned **err_word) { return current_device(err_word); }

int record_cuda_error(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    cudaGetLastError();   // do not leak a launch error into the caller's next check
    return GDA_ERR_CUDA;
}

bool encode_tmap_4d_bf16(CUtensorMap *map, const void *base, const uint64_t dims[4],
                         const uint64_t strides_bytes[3], const uint32_t box[4]) {
    std::call_once(g_encode_once, []() {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    if (!g_encode) return false;
    cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gstr[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    cuuint32_t bdim[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), gdim,
                                gstr, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace gda

using namespace gda;

extern "C" {

int gda_attn_fwd_ex(const void *q_sig, const void *k_sig, const void *q_noise, const void *k_noise,
                    const void *v, const float *lambda, float lambda_init, void *out, int B, int L,
                    int h_s, int h_n, int d, int dv, int causal, float eps, unsigned flags,
                    gda_stream_t stream) {
    int st = check_prefill_common(q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L,
                                  h_s, h_n, d, dv, causal, eps, flags,
                                  GDA_FLAG_NO_NORM | GDA_FLAG_SINGLE_PASS);
    if (st != GDA_OK) return st;
    if (!(d == 64 || d == 128) || !(dv == 128 || dv == 256)) return GDA_ERR_UNSUPPORTED;
    unsigned *err = nullptr;
    st = current_device(&err);
    if (st != GDA_OK) return st;
    PrefillArgs a{q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L, h_s, h_n,
                  d, dv, causal, eps, flags & GDA_FLAG_NO_NORM, err};
    if (!(flags & GDA_FLAG_SINGLE_PASS) && prefill_group_supported(a))
        return launch_prefill_group(a, reinterpret_cast<cudaStream_t>(stream));
    return launch_prefill_tc(a, reinterpret_cast<cudaStream_t>(stream));
}

int gda_attn_fwd_chunk(const void *q_sig, const void *k_sig, const void *q_noise, const void *k_noise,
                       const void *v, const float *lambda, float lambda_init, void *out, int B, int L,
                       int Lk, int h_s, int h_n, int d, int dv, int causal, float eps, unsigned flags,
                       gda_stream_t stream) {
    int st = check_prefill_common(q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L,
                                  h_s, h_n, d, dv, causal, eps, flags,
                                  GDA_FLAG_NO_NORM | GDA_FLAG_SINGLE_PASS);
    if (st != GDA_OK) return st;
    if (Lk < 1 || (causal && Lk < L)) return GDA_ERR_INVALID_ARG;
    if (static_cast<double>(B) * Lk * (h_s > h_n ? h_s : h_n) * (d > dv ? d : dv) > 9.0e15)
        return GDA_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128) || !(dv == 128 || dv == 256)) return GDA_ERR_UNSUPPORTED;
    unsigned *err = nullptr;
    st = current_device(&err);
    if (st != GDA_OK) return st;
    PrefillArgs a{q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L, h_s, h_n,
                  d, dv, causal, eps, flags & GDA_FLAG_NO_NORM, err};
    a.Lk = Lk;
    if (!(flags & GDA_FLAG_SINGLE_PASS) && prefill_group_supported(a))
        return launch_prefill_group(a, reinterpret_cast<cudaStream_t>(stream));
    return launch_prefill_tc(a, reinterpret_cast<cudaStream_t>(stream));
}

int gda_attn_fwd_chunk_2pass(const void *q_sig, const void *k_sig, const void *q_noise, const void *k_noise,
                             const void *v, const float *lambda, float lambda_init, void *out, int B, int L,
                             int Lk, int h_s, int h_n, int d, int dv, int causal, float eps, unsigned flags,
                             void *workspace, size_t workspace_bytes, gda_stream_t stream) {
    int st = check_prefill_common(q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L,
                                  h_s, h_n, d, dv, causal, eps, flags);
    if (st != GDA_OK) return st;
    if (Lk < 1 || (causal && Lk < L)) return GDA_ERR_INVALID_ARG;
    if (static_cast<double>(B) * Lk * (h_s > h_n ? h_s : h_n) * (d > dv ? d : dv) > 9.0e15)
        return GDA_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128) || !(dv == 128 || dv == 256)) return GDA_ERR_UNSUPPORTED;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < prefill_2pass_workspace_bytes(B, L, h_s, h_n))
        return GDA_ERR_WORKSPACE;
    unsigned *err = nullptr;
    st = current_device(&err);
    if (st != GDA_OK) return st;
    PrefillArgs a{q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L, h_s, h_n,
                  d, dv, causal, eps, flags, err};
    a.Lk = Lk;
    return launch_prefill_2pass(a, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int gda_attn_fwd(const void *q_sig, const void *k_sig, const void *q_noise, const void *k_noise,
                 const void *v, const float *lambda, float lambda_init, void *out, int B, int L,
                 int h_s, int h_n, int d, int dv, int causal, float eps, gda_stream_t stream) {
    return gda_attn_fwd_ex(q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L, h_s,
                           h_n, d, dv, causal, eps, 0u, stream);
}

int gda_attn_fwd_f32_ex(const float *q_sig, const float *k_sig, const float *q_noise,
                        const float *k_noise, const float *v, const float *lambda,
                        float lambda_init, float *out, int B, int L, int h_s, int h_n, int d,
                        int dv, int causal, float eps, unsigned flags, gda_stream_t stream) {
    int st = check_prefill_common(q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L,
                                  h_s, h_n, d, dv, causal, eps, flags);
    if (st != GDA_OK) return st;
    if (d > 256 || dv % 32 != 0 || dv > 256) return GDA_ERR_UNSUPPORTED;
    if (h_s > 65535 || B > 65535) return GDA_ERR_UNSUPPORTED;
    unsigned *err = nullptr;
    st = current_device(&err);
    if (st != GDA_OK) return st;
    PrefillArgs a{q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L, h_s, h_n,
                  d, dv, causal, eps, flags, err};
    return launch_prefill_f32(a, reinterpret_cast<cudaStream_t>(stream));
}

int gda_attn_fwd_f32(const float *q_sig, const float *k_sig, const float *q_noise,
                     const float *k_noise, const float *v, const float *lambda, float lambda_init,
                     float *out, int B, int L, int h_s, int h_n, int d, int dv, int causal,
                     float eps, gda_stream_t stream) {
    return gda_attn_fwd_f32_ex(q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L,
                               h_s, h_n, d, dv, causal, eps, 0u, stream);
}

size_t gda_attn_bwd_bf16_workspace_size(int B, int L, int h_s, int h_n, int dv) {
    if (B < 1 || L < 1 || h_s < 1 || h_n < 1 || dv < 1) return 0;
    if (static_cast<double>(B) * L * (h_s + h_n) * (dv > 1 ? dv : 1) > 9.0e15) return 0;
    return backward_tc_workspace_bytes(B, L, h_s, h_n, dv);
}

int gda_attn_bwd_bf16(const void *q_sig, const void *k_sig, const void *q_noise, const void *k_noise,
                      const void *v, const float *lambda, float lambda_init, const void *dy, float *dq_sig,
                      float *dk_sig, float *dq_noise, float *dk_noise, float *dv_out, float *dlambda, int B,
                      int L, int h_s, int h_n, int d, int dv, int causal, float eps, unsigned flags,
                      void *workspace, size_t workspace_bytes, gda_stream_t stream) {
    int st = check_prefill_common(q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, dy, B, L, h_s,
                                  h_n, d, dv, causal, eps, flags);
    if (st != GDA_OK) return st;
    if (!dq_sig || !dk_sig || !dq_noise || !dk_noise || !dv_out || !dlambda) return GDA_ERR_INVALID_ARG;
    if (d != 64 || dv != 128) return GDA_ERR_UNSUPPORTED;
    if (!aligned16(dq_sig) || !aligned16(dk_sig) || !aligned16(dq_noise) || !aligned16(dk_noise) ||
        !aligned16(dv_out) || !aligned16(dlambda))
        return GDA_ERR_MISALIGNED;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < gda_attn_bwd_bf16_workspace_size(B, L, h_s, h_n, dv))
        return GDA_ERR_WORKSPACE;
    unsigned *err = nullptr;
    st = current_device(&err);
    if (st != GDA_OK) return st;
    BackwardTcArgs a{q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, dy, dq_sig, dk_sig, dq_noise,
                     dk_noise, dv_out, dlambda, B, L, h_s, h_n, d, dv, causal, eps, flags, workspace, err};
    return launch_backward_tc(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t gda_attn_fwd_2pass_workspace_size(int B, int L, int h_s, int h_n) {
    if (B < 1 || L < 1 || h_s < 1 || h_n < 1) return 0;
    if (static_cast<double>(B) * L * (h_s + h_n) > 9.0e15) return 0;
    return prefill_2pass_workspace_bytes(B, L, h_s, h_n);
}

int gda_attn_fwd_2pass(const void *q_sig, const void *k_sig, const void *q_noise, const void *k_noise,
                       const void *v, const float *lambda, float lambda_init, void *out, int B, int L,
                       int h_s, int h_n, int d, int dv, int causal, float eps, unsigned flags,
                       void *workspace, size_t workspace_bytes, gda_stream_t stream) {
    int st = check_prefill_common(q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L,
                                  h_s, h_n, d, dv, causal, eps, flags);
    if (st != GDA_OK) return st;
    if (!(d == 64 || d == 128) || !(dv == 128 || dv == 256)) return GDA_ERR_UNSUPPORTED;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < gda_attn_fwd_2pass_workspace_size(B, L, h_s, h_n))
        return GDA_ERR_WORKSPACE;
    unsigned *err = nullptr;
    st = current_device(&err);
    if (st != GDA_OK) return st;
    PrefillArgs a{q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, out, B, L, h_s, h_n,
                  d, dv, causal, eps, flags, err};
    return launch_prefill_2pass(a, workspace, reinterpret_cast<cudaStream_t>(stream));
}

size_t gda_attn_bwd_workspace_size(int B, int L, int h_s, int d, int dv) {
    if (B < 1 || L < 1 || h_s < 1 || d < 1 || dv < 1) return 0;
    if (static_cast<double>(B) * L * h_s * (d > dv ? d : dv) > 9.0e15) return 0;
    return backward_f32_workspace_bytes(B, L, h_s, d, dv);
}

int gda_attn_bwd(const float *q_sig, const float *k_sig, const float *q_noise, const float *k_noise,
                 const float *v, const float *lambda, float lambda_init, const float *dy, float *dq_sig,
                 float *dk_sig, float *dq_noise, float *dk_noise, float *dv_out, float *dlambda, int B,
                 int L, int h_s, int h_n, int d, int dv, int causal, float eps, unsigned flags,
                 void *workspace, size_t workspace_bytes, gda_stream_t stream) {
    int st = check_prefill_common(q_sig, k_sig, q_noise, k_noise, v, lambda, lambda_init, dy, B, L, h_s,
                                  h_n, d, dv, causal, eps, flags);
    if (st != GDA_OK) return st;
    if (!dq_sig || !dk_sig || !dq_noise || !dk_noise || !dv_out || !dlambda) return GDA_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128) || !(dv == 64 || dv == 128 || dv == 256)) return GDA_ERR_UNSUPPORTED;
    if (h_s > 65535 || B > 65535) return GDA_ERR_UNSUPPORTED;
    if (!aligned16(dq_sig) || !aligned16(dk_sig) || !aligned16(dq_noise) || !aligned16(dk_noise) ||
        !aligned16(dv_out) || !aligned16(dlambda))
        return GDA_ERR_MISALIGNED;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < gda_attn_bwd_workspace_size(B, L, h_s, d, dv))
        return GDA_ERR_WORKSPACE;
    unsigned *err = nullptr;
    st = current_device(&err);
    if (st != GDA_OK) return st;
    BackwardArgs a{q_sig, k_sig, q_noise, k_noise, v, lambda, dy, lambda_init, dq_sig, dk_sig, dq_noise,
                   dk_noise, dv_out, dlambda, B, L, h_s, h_n, d, dv, causal, eps, flags, workspace};
    return launch_backward_f32(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t gda_attn_decode_workspace_size(int B, int Lcap, int h_s, int h_n, int dv) {
    if (B < 1 || Lcap < 1 || h_s < 1 || h_n < 1 || dv < 1 || h_s % h_n != 0) return 0;
    return decode_plan(B, Lcap, h_s, h_n, dv).bytes;
}

int gda_attn_decode(const void *q_sig, const void *q_noise, const void *k_sig_cache,
                    const void *k_noise_cache, const void *v_cache, const int *cache_lens,
                    const float *lambda, float lambda_init, void *out, int B, int Lcap, int h_s,
                    int h_n, int d, int dv, float eps, void *workspace, size_t workspace_bytes,
                    gda_stream_t stream) {
    if (!q_sig || !q_noise || !k_sig_cache || !k_noise_cache || !v_cache || !cache_lens || !lambda ||
        !out)
        return GDA_ERR_INVALID_ARG;
    if (B < 1 || Lcap < 1 || h_s < 1 || h_n < 1 || d < 1 || dv < 1 || h_s % h_n != 0)
        return GDA_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(lambda_init)) return GDA_ERR_INVALID_ARG;
    if (static_cast<double>(B) * Lcap * h_s * (d > dv ? d : dv) > 9.0e15) return GDA_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128) || !(dv == 64 || dv == 128 || dv == 256)) return GDA_ERR_UNSUPPORTED;
    if ((h_s * d + h_n * d + h_s * dv) / 8 > 1024 || h_s + h_n > 128 || B > 65535)
        return GDA_ERR_UNSUPPORTED;
    if (!aligned16(q_sig) || !aligned16(q_noise) || !aligned16(k_sig_cache) ||
        !aligned16(k_noise_cache) || !aligned16(v_cache) || !aligned16(cache_lens) ||
        !aligned16(lambda) || !aligned16(out))
        return GDA_ERR_MISALIGNED;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < gda_attn_decode_workspace_size(B, Lcap, h_s, h_n, dv))
        return GDA_ERR_WORKSPACE;
    unsigned *err = nullptr;
    const int st = current_device(&err);
    if (st != GDA_OK) return st;
    DecodeArgs a{q_sig, q_noise, k_sig_cache, k_noise_cache, v_cache, cache_lens, lambda, lambda_init,
                 out, B, Lcap, h_s, h_n, d, dv, eps, workspace, workspace_bytes, err};
    return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

int gda_attn_decode_fp8(const void *q_sig, const void *q_noise, const void *k_sig_cache,
                        const void *k_noise_cache, const void *v_cache, const float *k_sig_scale,
                        const float *k_noise_scale, const float *v_scale, const int *cache_lens,
                        const float *lambda, float lambda_init, void *out, int B, int Lcap, int h_s,
                        int h_n, int d, int dv, float eps, void *workspace, size_t workspace_bytes,
                        gda_stream_t stream) {
    if (!q_sig || !q_noise || !k_sig_cache || !k_noise_cache || !v_cache || !k_sig_scale || !k_noise_scale ||
        !v_scale || !cache_lens || !lambda || !out)
        return GDA_ERR_INVALID_ARG;
    if (B < 1 || Lcap < 1 || h_s < 1 || h_n < 1 || d < 1 || dv < 1 || h_s % h_n != 0)
        return GDA_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(lambda_init)) return GDA_ERR_INVALID_ARG;
    if (static_cast<double>(B) * Lcap * h_s * (d > dv ? d : dv) > 9.0e15) return GDA_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128) || !(dv == 64 || dv == 128 || dv == 256)) return GDA_ERR_UNSUPPORTED;
    if (h_s + h_n > 128 || B > 65535) return GDA_ERR_UNSUPPORTED;
    if (!aligned16(q_sig) || !aligned16(q_noise) || !aligned16(k_sig_cache) || !aligned16(k_noise_cache) ||
        !aligned16(v_cache) || !aligned16(cache_lens) || !aligned16(lambda) || !aligned16(out))
        return GDA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(k_sig_scale) | reinterpret_cast<uintptr_t>(k_noise_scale) |
         reinterpret_cast<uintptr_t>(v_scale)) & 3u)
        return GDA_ERR_MISALIGNED;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < gda_attn_decode_workspace_size(B, Lcap, h_s, h_n, dv))
        return GDA_ERR_WORKSPACE;
    unsigned *err = nullptr;
    const int st = current_device(&err);
    if (st != GDA_OK) return st;
    DecodeArgs a{q_sig, q_noise, k_sig_cache, k_noise_cache, v_cache, cache_lens, lambda, lambda_init,
                 out, B, Lcap, h_s, h_n, d, dv, eps, workspace, workspace_bytes, err};
    a.fp8 = 1;
    a.k1_scale = k_sig_scale;
    a.k2_scale = k_noise_scale;
    a.v_scale = v_scale;
    return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

int gda_attn_decode_paged(const void *q_sig, const void *q_noise, const void *k_sig_pool,
                          const void *k_noise_pool, const void *v_pool, const int *block_table,
                          const int *cache_lens, const float *lambda, float lambda_init, void *out, int B,
                          int max_pages, int page_size, int num_pages, int h_s, int h_n, int d, int dv,
                          float eps, void *workspace, size_t workspace_bytes, gda_stream_t stream) {
    if (!q_sig || !q_noise || !k_sig_pool || !k_noise_pool || !v_pool || !block_table || !cache_lens ||
        !lambda || !out)
        return GDA_ERR_INVALID_ARG;
    if (B < 1 || max_pages < 1 || page_size < 1 || num_pages < 1 || h_s < 1 || h_n < 1 || d < 1 || dv < 1 ||
        h_s % h_n != 0)
        return GDA_ERR_INVALID_ARG;
    const long long Lcap = static_cast<long long>(max_pages) * page_size;
    if (Lcap > 0x7fffffffLL) return GDA_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(lambda_init)) return GDA_ERR_INVALID_ARG;
    if (static_cast<double>(num_pages) * page_size * h_s * (d > dv ? d : dv) > 9.0e15) return GDA_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128) || !(dv == 64 || dv == 128 || dv == 256)) return GDA_ERR_UNSUPPORTED;
    if ((h_s * d + h_n * d + h_s * dv) / 8 > 1024 || h_s + h_n > 128 || B > 65535) return GDA_ERR_UNSUPPORTED;
    if (!aligned16(q_sig) || !aligned16(q_noise) || !aligned16(k_sig_pool) || !aligned16(k_noise_pool) ||
        !aligned16(v_pool) || !aligned16(cache_lens) || !aligned16(lambda) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u))
        return GDA_ERR_MISALIGNED;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < gda_attn_decode_workspace_size(B, static_cast<int>(Lcap), h_s, h_n, dv))
        return GDA_ERR_WORKSPACE;
    unsigned *err = nullptr;
    const int st = current_device(&err);
    if (st != GDA_OK) return st;
    DecodeArgs a{q_sig, q_noise, k_sig_pool, k_noise_pool, v_pool, cache_lens, lambda, lambda_init,
                 out, B, static_cast<int>(Lcap), h_s, h_n, d, dv, eps, workspace, workspace_bytes, err};
    a.block_table = block_table;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

int gda_attn_decode_paged_fp8(const void *q_sig, const void *q_noise, const void *k_sig_pool,
                              const void *k_noise_pool, const void *v_pool, const float *k_sig_scale,
                              const float *k_noise_scale, const float *v_scale, const int *block_table,
                              const int *cache_lens, const float *lambda, float lambda_init, void *out, int B,
                              int max_pages, int page_size, int num_pages, int h_s, int h_n, int d, int dv,
                              float eps, void *workspace, size_t workspace_bytes, gda_stream_t stream) {
    if (!q_sig || !q_noise || !k_sig_pool || !k_noise_pool || !v_pool || !k_sig_scale || !k_noise_scale ||
        !v_scale || !block_table || !cache_lens || !lambda || !out)
        return GDA_ERR_INVALID_ARG;
    if (B < 1 || max_pages < 1 || page_size < 1 || num_pages < 1 || h_s < 1 || h_n < 1 || d < 1 || dv < 1 ||
        h_s % h_n != 0)
        return GDA_ERR_INVALID_ARG;
    const long long Lcap = static_cast<long long>(max_pages) * page_size;
    if (Lcap > 0x7fffffffLL) return GDA_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(lambda_init)) return GDA_ERR_INVALID_ARG;
    if (static_cast<double>(num_pages) * page_size * h_s * (d > dv ? d : dv) > 9.0e15) return GDA_ERR_INVALID_ARG;
    if (!(d == 64 || d == 128) || !(dv == 64 || dv == 128 || dv == 256)) return GDA_ERR_UNSUPPORTED;
    if (h_s + h_n > 128 || B > 65535) return GDA_ERR_UNSUPPORTED;
    if (!aligned16(q_sig) || !aligned16(q_noise) || !aligned16(k_sig_pool) || !aligned16(k_noise_pool) ||
        !aligned16(v_pool) || !aligned16(cache_lens) || !aligned16(lambda) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u))
        return GDA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(k_sig_scale) | reinterpret_cast<uintptr_t>(k_noise_scale) |
         reinterpret_cast<uintptr_t>(v_scale)) & 3u)
        return GDA_ERR_MISALIGNED;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < gda_attn_decode_workspace_size(B, static_cast<int>(Lcap), h_s, h_n, dv))
        return GDA_ERR_WORKSPACE;
    unsigned *err = nullptr;
    const int st = current_device(&err);
    if (st != GDA_OK) return st;
    DecodeArgs a{q_sig, q_noise, k_sig_pool, k_noise_pool, v_pool, cache_lens, lambda, lambda_init,
                 out, B, static_cast<int>(Lcap), h_s, h_n, d, dv, eps, workspace, workspace_bytes, err};
    a.fp8 = 1;
    a.k1_scale = k_sig_scale;
    a.k2_scale = k_noise_scale;
    a.v_scale = v_scale;
    a.block_table = block_table;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

int gda_lambda_reparam(const float *lambda_q1, const float *lambda_k1, const float *lambda_q2,
                       const float *lambda_k2, float lambda_init, float *lambda_out, int h_s, int d,
                       gda_stream_t stream) {
    if (!lambda_q1 || !lambda_k1 || !lambda_q2 || !lambda_k2 || !lambda_out) return GDA_ERR_INVALID_ARG;
    if (h_s < 1 || d < 1 || !std::isfinite(lambda_init)) return GDA_ERR_INVALID_ARG;
    if (static_cast<long long>(h_s) * d > 0x7fffffffLL) return GDA_ERR_INVALID_ARG;
    const uintptr_t any = reinterpret_cast<uintptr_t>(lambda_q1) | reinterpret_cast<uintptr_t>(lambda_k1) |
                          reinterpret_cast<uintptr_t>(lambda_q2) | reinterpret_cast<uintptr_t>(lambda_k2) |
                          reinterpret_cast<uintptr_t>(lambda_out);
    if (any & 3u) return GDA_ERR_MISALIGNED;
    unsigned *err = nullptr;
    const int st = current_device(&err);
    if (st != GDA_OK) return st;
    return launch_lambda_reparam(lambda_q1, lambda_k1, lambda_q2, lambda_k2, lambda_init, lambda_out, h_s, d,
                                 reinterpret_cast<cudaStream_t>(stream));
}

const char *gda_status_string(int status) {
    switch (status) {
        case GDA_OK: return "success";
        case GDA_ERR_INVALID_ARG: return "invalid argument";
        case GDA_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case GDA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case GDA_ERR_WORKSPACE: return "workspace missing or too small";
        case GDA_ERR_CUDA: return "CUDA runtime or driver error";
        case GDA_ERR_DEVICE_TIMEOUT: return "a kernel wait timed out";
        default: return "unknown status";
    }
}

int gda_last_cuda_error(void) { return g_last_cuda_error; }

int gda_device_error(int clear) {
    unsigned *err = nullptr;
    const int st = current_device(&err);
    if (st != GDA_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GDA_ERR_CUDA;
    }
    unsigned v = 0;
    if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return GDA_ERR_CUDA;
    }
    if (clear && cudaMemset(err, 0, sizeof(unsigned)) != cudaSuccess) {
        cudaGetLastError();
        return GDA_ERR_CUDA;
    }
    return static_cast<int>(v & 0x7fffffffu);
}

}  // extern "C"
