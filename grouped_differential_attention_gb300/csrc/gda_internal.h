// Internal host-side interface between the C ABI (gda_api.cu) and the kernel
// translation units.  Not installed, not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace gda {

struct PrefillArgs {
    const void *q1, *k1, *q2, *k2, *v;   // see include/gda.h for layouts
    const float *lambda;
    float lambda_init;
    void *out;
    int B, L, hs, hn, d, dv;
    int causal;
    float eps;
    unsigned flags;
    unsigned *dev_err;                  // device error word of the current device
    int Lk = 0;                         // keys per sequence (0: L); query row i is key position Lk - L + i
};

struct DecodeArgs {
    const void *q1, *q2, *k1c, *k2c, *vc;
    const int *lens;
    const float *lambda;
    float lambda_init;
    void *out;
    int B, Lcap, hs, hn, d, dv;
    float eps;
    void *workspace;
    size_t workspace_bytes;
    unsigned *dev_err;
    int fp8 = 0;                                  // caches hold fp8 (e4m3) codes
    const int *block_table = nullptr;             // paged caches (see gda_attn_decode_paged)
    int page_size = 0, max_pages = 0, num_pages = 0;
    const float *k1_scale = nullptr, *k2_scale = nullptr, *v_scale = nullptr;
};

struct BackwardArgs {
    const float *q1, *k1, *q2, *k2, *v, *lambda, *dy;   // float32, layouts of gda_attn_fwd
    float lambda_init;
    float *dq1, *dk1, *dq2, *dk2, *dv_out, *dlambda;
    int B, L, hs, hn, d, dv;
    int causal;
    float eps;
    unsigned flags;
    void *workspace;
};

struct BackwardTcArgs {
    const void *q1, *k1, *q2, *k2, *v;   // bf16, layouts of gda_attn_fwd
    const float *lambda;
    float lambda_init;
    const void *dy;                      // bf16 [B, L, hs, dv]
    float *dq1, *dk1, *dq2, *dk2, *dv_out, *dlambda;
    int B, L, hs, hn, d, dv;
    int causal;
    float eps;
    unsigned flags;
    void *workspace;
    unsigned *dev_err;
};

// Remembers `e` as this thread's last CUDA error (see gda_last_cuda_error),
// clears the runtime's sticky-free error state and returns GDA_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Checks the current device (GB300, compute capability 10.3) once and
// returns a gda_status plus the address of its device error word.
int device_state(unsigned **err_word);

// Each launcher validates nothing (the ABI layer did) and returns a
// gda_status value.
int launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream);
// The grouped kernel (noise map once per noise head and query tile): d = 64, dv = 128.
bool prefill_group_supported(const PrefillArgs &a);
int launch_prefill_group(const PrefillArgs &a, cudaStream_t stream);
int launch_prefill_f32(const PrefillArgs &a, cudaStream_t stream);
int launch_decode(const DecodeArgs &a, cudaStream_t stream);
int launch_prefill_2pass(const PrefillArgs &a, void *workspace, cudaStream_t stream);
size_t prefill_2pass_workspace_bytes(int B, int L, int hs, int hn);
// Pass 1 alone: base-2 log-sum-exp of every signal and noise map row into
// lse [B, hs + hn, lse_ld] (lse_ld >= L).
int launch_lse_pass(const PrefillArgs &a, float *lse, int lse_ld, cudaStream_t stream);
int launch_backward_f32(const BackwardArgs &a, cudaStream_t stream);
int launch_backward_tc(const BackwardTcArgs &a, cudaStream_t stream);
size_t backward_tc_workspace_bytes(int B, int L, int hs, int hn, int dv);
size_t backward_f32_workspace_bytes(int B, int L, int hs, int d, int dv);
int launch_lambda_reparam(const float *lq1, const float *lk1, const float *lq2, const float *lk2,
                          float lambda_init, float *out, int hs, int d, cudaStream_t stream);

// Split plan of the decode kernel (positions per split and split count).
struct DecodePlan {
    int slots;        // partial-state slots (split CTAs + sequences)
    size_t o_bytes;   // accumulator partials
    size_t ml_bytes;  // (max, sum) partials
    size_t bytes;     // workspace bytes
};
DecodePlan decode_plan(int B, int Lcap, int hs, int hn, int dv);

// 4-D bf16 tensor map, 128-byte swizzle, dims/box innermost first, strides
// in bytes for dims 1..3.  Returns false if the driver rejects it.
bool encode_tmap_4d_bf16(CUtensorMap *map, const void *base, const uint64_t dims[4],
                         const uint64_t strides_bytes[3], const uint32_t box[4]);

}  // namespace gda
