/*
 * gda.h -- C ABI of the grouped differential attention library (libgda.so)
 * for NVIDIA GB300 (sm_103a).
 *
 * THE OPERATION
 *   Grouped differential attention ("Grouped Differential Attention",
 *   arXiv 2510.06949, abstract) splits the heads of a layer into h_s signal
 *   heads and h_n <= h_s noise-control heads, h_s a multiple of h_n.  Noise
 *   head g is shared by the r = h_s / h_n consecutive signal heads
 *   h = g*r .. g*r + r - 1 (grouped-query style repetition).  For signal head h
 *   with noise head g = h / r it computes, per query row,
 *
 *     o_h = ( softmax(Q1_h K1_h^T / sqrt(d)) - lambda_h * softmax(Q2_g K2_g^T / sqrt(d)) ) V_h
 *     y_h = (1 - lambda_init) * o_h / sqrt(mean_over_dv(o_h^2) + eps)
 *
 *   which is the differential attention operator and its headwise
 *   normalisation of "Differential Attention in Large Language Models: How
 *   Denoising Subtraction Eliminates Attention Noise and Outlier
 *   Activations" (sections "Differential Attention Architecture" and
 *   "Headwise Normalization"), with the second map taken from the shared
 *   noise head.  With h_s == h_n it is plain differential attention.  The
 *   RMSNorm has no learnable gain.  Both softmaxes are normalised before the
 *   subtraction; the subtraction and the norm are done in float32.
 *
 * LAYOUT (all tensors dense, row-major, innermost dimension last)
 *   q_sig, k_sig : [B, L, h_s, d]      signal queries / keys   (Q1, K1)
 *   q_noise, k_noise : [B, L, h_n, d]  noise queries / keys    (Q2, K2)
 *   v            : [B, L, h_s, dv]     values (dv is the 2d of the pages)
 *   lambda       : [h_s] float32       per signal head; a layer-wide lambda
 *                                      is the case of equal entries
 *   out          : [B, L, h_s, dv]     same dtype as the inputs
 *   Causal masking lets query i see keys 0..i.
 *
 * OWNERSHIP AND ASYNCHRONY
 *   Every pointer is owned by the caller and must stay valid until the work
 *   enqueued on `stream` has finished.  Device pointers must be device
 *   memory of the current CUDA device.  The library allocates no device
 *   memory in these calls; the decode call uses the caller's workspace.  Calls
 *   only enqueue work on `stream` (NULL = the legacy default stream) and
 *   return; kernel faults surface at the caller's next synchronisation.
 *   The library keeps per-device state: a device error word (see
 *   gda_device_error) and cached driver entry points.
 *
 * ERRORS
 *   Every call returns a gda_status.  Arguments are validated before any
 *   CUDA call is made; invalid arguments return without enqueuing work.
 *   Nothing is thrown across the ABI.
 */
#ifndef GDA_H
#define GDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *gda_stream_t;

typedef enum {
    GDA_OK = 0,
    GDA_ERR_INVALID_ARG = -1,    /* null pointer, non-positive size, h_s % h_n != 0, ... */
    GDA_ERR_UNSUPPORTED = -2,    /* valid but not implemented: head dims, device arch */
    GDA_ERR_MISALIGNED = -3,     /* a pointer is not 16-byte aligned */
    GDA_ERR_WORKSPACE = -4,      /* decode workspace null or too small */
    GDA_ERR_CUDA = -5,           /* a CUDA runtime/driver call failed (incl. no device) */
    GDA_ERR_DEVICE_TIMEOUT = -6  /* a kernel gave up waiting (see gda_device_error) */
} gda_status;

/* Flags for the *_ex entry points. */
#define GDA_FLAG_NO_NORM 0x1u    /* return o_h (pre-norm, float32 difference) instead of y_h */
#define GDA_FLAG_SINGLE_PASS 0x2u /* gda_attn_fwd_ex, gda_attn_fwd_chunk: run the per-signal-head single-pass kernel */

/*
 * Prefill / full-sequence forward, bf16 I/O, float32 accumulation.
 *   Inputs and out: bf16 device tensors in the layout above.
 *   lambda: float32 device array [h_s].
 *   Supported: d in {64, 128}; dv in {128, 256}; B, L >= 1; h_s % h_n == 0;
 *   every pointer 16-byte aligned; device sm_103 (GB300).  causal in {0, 1}.
 *   Output is rounded once to bf16 (round to nearest even).
 * Computed by hand-written tcgen05/TMA kernels in one pass with two running
 * softmax states per row; no workspace and no allocation (at dv = 256 the
 * 256 accumulator columns are split over a CTA pair).  Callers that can
 * provide a workspace get the faster two-pass kernels at dv = 256 from
 * gda_attn_fwd_2pass.
 */
int gda_attn_fwd(const void *q_sig, const void *k_sig, const void *q_noise,
                 const void *k_noise, const void *v, const float *lambda,
                 float lambda_init, void *out, int B, int L, int h_s, int h_n,
                 int d, int dv, int causal, float eps, gda_stream_t stream);

/*
 * Chunked prefill: L new query rows continuing a sequence whose keys and
 * values (the cached prefix plus the chunk itself) are Lk >= L rows long.
 * Query row i sits at key position Lk - L + i and, when causal, attends keys
 * 0 .. Lk - L + i; non-causal, all Lk keys.  The result equals the last L
 * rows of gda_attn_fwd over the whole Lk-row sequence.  (Prefill that
 * continues from a cache is on the serving path of "Hardware Implementations
 * and Serving Considerations".)
 *   q_sig [B, L, h_s, d], q_noise [B, L, h_n, d], out [B, L, h_s, dv];
 *   k_sig [B, Lk, h_s, d], k_noise [B, Lk, h_n, d], v [B, Lk, h_s, dv].
 * Other arguments, flags, kernels (no workspace, no allocation), support and
 * errors as gda_attn_fwd_ex; GDA_ERR_INVALID_ARG also for Lk < 1 or (causal
 * and Lk < L).
 */
int gda_attn_fwd_chunk(const void *q_sig, const void *k_sig, const void *q_noise, const void *k_noise,
                       const void *v, const float *lambda, float lambda_init, void *out, int B, int L,
                       int Lk, int h_s, int h_n, int d, int dv, int causal, float eps, unsigned flags,
                       gda_stream_t stream);

/*
 * Chunked prefill through the two-pass kernels of gda_attn_fwd_2pass (the
 * faster choice at dv = 256).  Arguments as gda_attn_fwd_chunk plus a
 * caller-owned device workspace of at least
 * gda_attn_fwd_2pass_workspace_size(B, L, h_s, h_n) bytes (L = the chunk's
 * query rows; 16-byte aligned), which receives the chunk rows' base-2
 * log-sum-exp values.  Flags: GDA_FLAG_NO_NORM.  GDA_ERR_WORKSPACE if the
 * workspace is null, misaligned or too small.
 */
int gda_attn_fwd_chunk_2pass(const void *q_sig, const void *k_sig, const void *q_noise, const void *k_noise,
                             const void *v, const float *lambda, float lambda_init, void *out, int B, int L,
                             int Lk, int h_s, int h_n, int d, int dv, int causal, float eps, unsigned flags,
                             void *workspace, size_t workspace_bytes, gda_stream_t stream);

/* gda_attn_fwd with flags (GDA_FLAG_NO_NORM, GDA_FLAG_SINGLE_PASS). */
int gda_attn_fwd_ex(const void *q_sig, const void *k_sig, const void *q_noise,
                    const void *k_noise, const void *v, const float *lambda,
                    float lambda_init, void *out, int B, int L, int h_s, int h_n,
                    int d, int dv, int causal, float eps, unsigned flags,
                    gda_stream_t stream);

/*
 * Prefill with float32 I/O and float32 arithmetic on the CUDA cores.
 *   Same layout and meaning as gda_attn_fwd, every tensor float32.
 *   Supported: 1 <= d <= 256; dv in {32, 64, ..., 256} (multiple of 32).
 */
int gda_attn_fwd_f32(const float *q_sig, const float *k_sig, const float *q_noise,
                     const float *k_noise, const float *v, const float *lambda,
                     float lambda_init, float *out, int B, int L, int h_s, int h_n,
                     int d, int dv, int causal, float eps, gda_stream_t stream);

/* gda_attn_fwd_f32 with flags (GDA_FLAG_NO_NORM). */
int gda_attn_fwd_f32_ex(const float *q_sig, const float *k_sig, const float *q_noise,
                        const float *k_noise, const float *v, const float *lambda,
                        float lambda_init, float *out, int B, int L, int h_s, int h_n,
                        int d, int dv, int causal, float eps, unsigned flags,
                        gda_stream_t stream);

/*
 * Two-pass bf16 prefill: the same operation and layouts as gda_attn_fwd_ex,
 * computed with the difference map formed before the value product
 * (o = (A1 - lambda_h A2) V_h; Differential Transformer, section
 * "Differential Attention": both maps are normalised softmax maps, so their
 * difference is fixed once each row's softmax statistics are known).
 *   Pass 1 writes each query row's base-2 log-sum-exp of every signal map
 *   (per signal head) and every noise map (once per noise head) to
 *   `workspace`; pass 2 recomputes the logits, forms P = A1 - lambda_h A2
 *   in float32, rounds it once to bf16 and runs one P V product per head into
 *   one float32 accumulator, then applies the headwise norm.
 *   workspace: device memory of at least gda_attn_fwd_2pass_workspace_size(
 *   B, L, h_s, h_n) bytes (float32 [B, h_s + h_n, L]), 16-byte aligned,
 *   owned by the caller; on return it holds the log-sum-exp values.
 *   Supported: d in {64, 128}, dv in {128, 256} (dv = 256 in one CTA).
 *   Returns as gda_attn_fwd_ex, plus GDA_ERR_WORKSPACE.
 */
int gda_attn_fwd_2pass(const void *q_sig, const void *k_sig, const void *q_noise,
                       const void *k_noise, const void *v, const float *lambda,
                       float lambda_init, void *out, int B, int L, int h_s, int h_n,
                       int d, int dv, int causal, float eps, unsigned flags,
                       void *workspace, size_t workspace_bytes, gda_stream_t stream);

/* Bytes of workspace gda_attn_fwd_2pass needs (0 for invalid sizes). */
size_t gda_attn_fwd_2pass_workspace_size(int B, int L, int h_s, int h_n);

/*
 * Backward (gradients) of the float32 operation above: given dy = dL/dy
 * (dL/do with GDA_FLAG_NO_NORM), the gradients of L with respect to the
 * signal and noise projections, the values and lambda.  Chain rule through
 * the two softmax maps (Differential Transformer, section "Differential
 * Attention"), the shared noise heads of a group (Grouped Differential
 * Attention, abstract and method: dq_noise and dk_noise sum over the h_s/h_n
 * signal heads that read each noise head) and the headwise RMSNorm (section
 * "Headwise Normalization", scale 1 - lambda_init, no learned gain).
 *   Inputs: the float32 tensors of gda_attn_fwd_f32 plus dy [B, L, h_s, dv].
 *   Outputs (float32 device, overwritten, no accumulation into them):
 *     dq_sig, dk_sig [B, L, h_s, d]; dq_noise, dk_noise [B, L, h_n, d];
 *     dv_out [B, L, h_s, dv]; dlambda [h_s] (summed over batch and rows).
 *   Supported: d in {64, 128}, dv in {64, 128, 256}.
 *   workspace: device memory of at least gda_attn_bwd_workspace_size(B, L,
 *   h_s, d, dv) bytes, 16-byte aligned, owned by the caller, not read across
 *   calls (holds each row's softmax statistics, dL/do and per-signal-head
 *   shares of the noise gradients).
 *   The forward is recomputed from the inputs (no forward state is passed).
 *   Results are deterministic (fixed summation orders).
 *   Returns GDA_OK, GDA_ERR_INVALID_ARG, GDA_ERR_UNSUPPORTED,
 *   GDA_ERR_MISALIGNED, GDA_ERR_WORKSPACE or GDA_ERR_CUDA; all argument
 *   checks run before any device work.
 */
int gda_attn_bwd(const float *q_sig, const float *k_sig, const float *q_noise,
                 const float *k_noise, const float *v, const float *lambda,
                 float lambda_init, const float *dy, float *dq_sig, float *dk_sig,
                 float *dq_noise, float *dk_noise, float *dv_out, float *dlambda,
                 int B, int L, int h_s, int h_n, int d, int dv, int causal,
                 float eps, unsigned flags, void *workspace,
                 size_t workspace_bytes, gda_stream_t stream);

/* Bytes of workspace gda_attn_bwd needs (0 for invalid sizes). */
size_t gda_attn_bwd_workspace_size(int B, int L, int h_s, int d, int dv);

/*
 * Backward on the tensor cores: the gradients of gda_attn_bwd (same
 * definitions, outputs, layouts and determinism) from bf16 inputs q_sig,
 * k_sig, q_noise, k_noise, v and dy (layouts of gda_attn_fwd; dy [B, L, h_s,
 * dv]); float32 lambda and float32 outputs.  Supported: d = 64, dv = 128.
 * The maps' row statistics are recomputed (no forward state is passed); the
 * norm's input gradient do is formed in float32 and rounded once to bf16,
 * W = A1 - lambda A2, dS1 and dS2 are rounded to bf16 as tensor-core
 * operands; every product accumulates in float32.  No atomics: each noise
 * head's gradients accumulate over its group in one CTA.
 *   workspace: device memory of at least gda_attn_bwd_bf16_workspace_size(B,
 *   L, h_s, h_n, dv) bytes, 16-byte aligned, owned by the caller (row
 *   statistics, do in bf16, D1 and D2).
 *   Returns as gda_attn_bwd.
 */
int gda_attn_bwd_bf16(const void *q_sig, const void *k_sig, const void *q_noise,
                      const void *k_noise, const void *v, const float *lambda,
                      float lambda_init, const void *dy, float *dq_sig, float *dk_sig,
                      float *dq_noise, float *dk_noise, float *dv_out, float *dlambda,
                      int B, int L, int h_s, int h_n, int d, int dv, int causal,
                      float eps, unsigned flags, void *workspace,
                      size_t workspace_bytes, gda_stream_t stream);

/* Bytes of workspace gda_attn_bwd_bf16 needs (0 for invalid sizes). */
size_t gda_attn_bwd_bf16_workspace_size(int B, int L, int h_s, int h_n, int dv);

/*
 * Bytes of device workspace gda_attn_decode needs for these sizes (it holds
 * the partial softmax states of the cache segments that the split kernel's
 * CTAs produce; the size does not depend on Lcap).  Returns 0 for invalid
 * sizes.
 */
size_t gda_attn_decode_workspace_size(int B, int Lcap, int h_s, int h_n, int dv);

/*
 * Decode: one new query token per sequence attends over its key/value cache
 * (the operation above for the last row of a causal prefill; the caller has
 * already appended the new token, so sequence b attends to cache rows
 * 0 .. cache_lens[b]-1).
 *   q_sig [B, h_s, d], q_noise [B, h_n, d]                       bf16
 *   k_sig_cache [B, Lcap, h_s, d], k_noise_cache [B, Lcap, h_n, d],
 *   v_cache [B, Lcap, h_s, dv]                                   bf16
 *   cache_lens [B] int32 device array, 1 <= cache_lens[b] <= Lcap
 *   lambda [h_s] float32 device; out [B, h_s, dv] bf16.
 *   workspace: device memory of at least
 *   gda_attn_decode_workspace_size(B, Lcap, h_s, h_n, dv) bytes, 16-byte
 *   aligned, owned by the caller; its contents need no initialisation.
 *   Two decode calls that are in flight at the same time need two
 *   workspaces.  A length outside [1, Lcap] is clamped on the device and
 *   reported through gda_device_error (GDA_DEVERR_BAD_LENGTH).
 *   Supported: d in {64, 128}; dv in {64, 128, 256}; h_s + h_n <= 128;
 *   32 + up32((h_s + h_n)*d/8) + up32(h_s*dv/8) <= 1024, up32 rounding up
 *   to a multiple of 32 (one thread per 16 bytes of a cache row, plus a
 *   producer warp).
 * Split kernel (the batch's cache positions cut into equal contiguous ranges,
 * one per CTA, streamed through shared memory by bulk copies) plus a
 * combine kernel.
 */
int gda_attn_decode(const void *q_sig, const void *q_noise, const void *k_sig_cache,
                    const void *k_noise_cache, const void *v_cache, const int *cache_lens,
                    const float *lambda, float lambda_init, void *out, int B, int Lcap,
                    int h_s, int h_n, int d, int dv, float eps, void *workspace,
                    size_t workspace_bytes, gda_stream_t stream);

/*
 * Decode over an fp8 cache ("Hardware Implementations and Serving
 * Considerations": low-bit KV cache quantisation on the serving path).
 * Same operation, layouts and workspace as gda_attn_decode, except:
 *   k_sig_cache, k_noise_cache, v_cache hold fp8 e4m3 codes (1 byte per
 *   element, same [B, Lcap, heads, dim] layout, 16-byte aligned); the cached
 *   value is code * scale of its head:
 *   k_sig_scale [h_s], k_noise_scale [h_n], v_scale [h_s]: float32 device
 *   arrays, 4-byte aligned.  Queries, lambda and the output stay as in
 *   gda_attn_decode (bf16 q, float32 lambda, bf16 out).
 * 2560 cache bytes per position for 12 + 4 heads, d = 64, dv = 128 (half of
 * bf16).  Supported: d in {64, 128}; dv in {64, 128, 256}; h_s + h_n <= 128;
 * 32 + up32((h_s + h_n) d / 16) + up32(h_s dv / 16) <= 1024.
 */
int gda_attn_decode_fp8(const void *q_sig, const void *q_noise, const void *k_sig_cache,
                        const void *k_noise_cache, const void *v_cache, const float *k_sig_scale,
                        const float *k_noise_scale, const float *v_scale, const int *cache_lens,
                        const float *lambda, float lambda_init, void *out, int B, int Lcap, int h_s,
                        int h_n, int d, int dv, float eps, void *workspace, size_t workspace_bytes,
                        gda_stream_t stream);

/*
 * Decode over paged caches (the paged KV layout of serving stacks; the pages
 * put the KV cache on the serving path, "Hardware Implementations and
 * Serving Considerations").  Same operation and result as gda_attn_decode;
 * the caches are page pools shared by all sequences:
 *   k_sig_pool [num_pages, page_size, h_s, d], k_noise_pool [num_pages,
 *   page_size, h_n, d], v_pool [num_pages, page_size, h_s, dv]      bf16
 *   block_table [B, max_pages] int32 device: cache position j of sequence b
 *   is row j % page_size of page block_table[b][j / page_size]
 *   cache_lens [B]: 1 <= cache_lens[b] <= max_pages * page_size
 * Workspace: gda_attn_decode_workspace_size(B, max_pages * page_size, h_s,
 * h_n, dv) bytes.  A block-table entry outside [0, num_pages) is read as page
 * 0 and reported through gda_device_error (GDA_DEVERR_BAD_PAGE).  Supported
 * sizes as gda_attn_decode; page_size >= 1.
 */
int gda_attn_decode_paged(const void *q_sig, const void *q_noise, const void *k_sig_pool,
                          const void *k_noise_pool, const void *v_pool, const int *block_table,
                          const int *cache_lens, const float *lambda, float lambda_init, void *out, int B,
                          int max_pages, int page_size, int num_pages, int h_s, int h_n, int d, int dv,
                          float eps, void *workspace, size_t workspace_bytes, gda_stream_t stream);

/*
 * Decode over paged fp8 (e4m3) caches: the page pools and block table of
 * gda_attn_decode_paged holding the e4m3 codes and per-head scales of
 * gda_attn_decode_fp8 (cached value = code x scale of its head).  Arguments,
 * layouts, ownership and errors as those two entries; both serving variants
 * ("Hardware Implementations and Serving Considerations": paged KV caches
 * and low-bit KV quantisation) at once.
 */
int gda_attn_decode_paged_fp8(const void *q_sig, const void *q_noise, const void *k_sig_pool,
                              const void *k_noise_pool, const void *v_pool, const float *k_sig_scale,
                              const float *k_noise_scale, const float *v_scale, const int *block_table,
                              const int *cache_lens, const float *lambda, float lambda_init, void *out, int B,
                              int max_pages, int page_size, int num_pages, int h_s, int h_n, int d, int dv,
                              float eps, void *workspace, size_t workspace_bytes, gda_stream_t stream);

/*
 * Decode that allocates nothing and takes no workspace.  No counterpart on
 * the pages: it exists for callers that cannot allocate device memory, such
 * as a plugin or serving loop whose host framework owns all device memory in
 * its own pool, or code that must not call cudaMalloc/cudaFree because those
 * calls can synchronise the device.
 *   Same arguments, layouts and result as gda_attn_decode, minus the
 *   workspace.  The split partials go to a scratch array inside the library,
 *   GDA_DECODE_SCRATCH_BYTES (32 MiB) per device, held by every device that
 *   loads the library until the process exits.
 *   Returns GDA_ERR_WORKSPACE if gda_attn_decode_workspace_size(B, Lcap, h_s,
 *   h_n, dv) exceeds GDA_DECODE_SCRATCH_BYTES (e.g. 64 sequences with
 *   12 + 4 heads and dv = 128 need about 8.3 MB whatever their lengths;
 *   more than about 2000 such sequences do not fit).
 *   The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  If the lookup fails the call returns
 *   GDA_ERR_CUDA and the next call on that device looks it up again.
 *   Every call shares the one array and it keeps the last call's contents
 *   (the kernels write every value they later read, so nothing needs
 *   clearing).  Calls whose work overlaps on the GPU, on any streams, race
 *   on the array and produce wrong results: serialise them.
 */
#define GDA_DECODE_SCRATCH_BYTES (32u << 20)
int gda_attn_decode_noalloc(const void *q_sig, const void *q_noise, const void *k_sig_cache,
                            const void *k_noise_cache, const void *v_cache, const int *cache_lens,
                            const float *lambda, float lambda_init, void *out, int B, int Lcap,
                            int h_s, int h_n, int d, int dv, float eps, gda_stream_t stream);

/*
 * Re-parameterised lambda of every signal head ("Differential Attention in
 * Large Language Models ...", section "Learnable Lambda Re-parameterization"):
 *   lambda_out[h] = exp(lambda_q1[h] . lambda_k1[h]) - exp(lambda_q2[h] . lambda_k2[h])
 *                   + lambda_init
 *   lambda_q1, lambda_k1, lambda_q2, lambda_k2: [h_s, d] float32 device arrays
 *   (one set of vectors per signal head; a per-layer lambda is the case of
 *   identical rows), 4-byte aligned, owned by the caller.
 *   lambda_out: [h_s] float32 device, the array gda_attn_fwd and
 *   gda_attn_decode take as lambda.  lambda_init: the layer's constant (for
 *   example 0.8 - 0.6 exp(-0.3 (l - 1)) for layer l).
 * float32 dot products (fused multiply-adds over d) and expf.  Enqueued on
 * `stream`; returns GDA_OK, GDA_ERR_INVALID_ARG (null pointer, h_s < 1,
 * d < 1, non-finite lambda_init), GDA_ERR_MISALIGNED or a device error.
 */
int gda_lambda_reparam(const float *lambda_q1, const float *lambda_k1, const float *lambda_q2,
                       const float *lambda_k2, float lambda_init, float *lambda_out, int h_s, int d,
                       gda_stream_t stream);

/* Static English description of a gda_status value. */
const char *gda_status_string(int status);

/*
 * cudaError_t value of the most recent CUDA failure that made a call of this
 * thread return GDA_ERR_CUDA (0 if none).  For diagnostics only.
 */
int gda_last_cuda_error(void);

/* Bits of the device error word. */
#define GDA_DEVERR_PREFILL_TIMEOUT 0x1u  /* a prefill pipeline wait ran out */
#define GDA_DEVERR_BAD_LENGTH      0x2u  /* a decode cache length was outside [1, Lcap] */
#define GDA_DEVERR_DECODE_TIMEOUT  0x4u  /* a decode cache-streaming wait ran out */
#define GDA_DEVERR_BAD_PAGE        0x8u  /* a paged decode's block table named a page outside the pool */

/*
 * Reads the error word of the current device (synchronises the device
 * first).  Kernels never trap: a pipeline wait that runs out (about one
 * second) sets a bit here and the kernel returns.  If clear != 0 the word is
 * reset to 0 after reading.  Returns the word (>= 0) or GDA_ERR_CUDA.
 */
int gda_device_error(int clear);

#ifdef __cplusplus
}
#endif

#endif /* GDA_H */
