// Re-parameterised lambda of every signal head on the device:
//   lambda_h = exp(lq1_h . lk1_h) - exp(lq2_h . lk2_h) + lambda_init
// ("Differential Attention in Large Language Models ...", section "Learnable
// Lambda Re-parameterization").  The result is the float32 [h_s] array the
// attention entry points take, so a training step never copies lambda
// through the host.
//
// One warp per head: lanes stride over the d components with fused
// multiply-adds, a shuffle reduction sums the lanes, lane 0 applies expf.
#include <cuda_runtime.h>
#include <cstdint>

#include "gda.h"
#include "gda_internal.h"

namespace gda {
namespace {

constexpr int kLambdaThreads = 128;   // four heads per block

__global__ void __launch_bounds__(kLambdaThreads)
gda_lambda_reparam_kernel(const float *__restrict__ lq1, const float *__restrict__ lk1,
                          const float *__restrict__ lq2, const float *__restrict__ lk2, float lambda_init,
                          float *__restrict__ out, int hs, int d) {
    const int h = blockIdx.x * (kLambdaThreads / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (h >= hs) return;                  // whole warp
    const size_t base = static_cast<size_t>(h) * d;
    float a = 0.f, b = 0.f;
    for (int i = lane; i < d; i += 32) {
        a = fmaf(lq1[base + i], lk1[base + i], a);
        b = fmaf(lq2[base + i], lk2[base + i], b);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if (lane == 0) out[h] = expf(a) - expf(b) + lambda_init;
}

}  // namespace

int launch_lambda_reparam(const float *lq1, const float *lk1, const float *lq2, const float *lk2,
                          float lambda_init, float *out, int hs, int d, cudaStream_t stream) {
    const int heads_per_block = kLambdaThreads / 32;
    const unsigned blocks = static_cast<unsigned>((hs + heads_per_block - 1) / heads_per_block);
    gda_lambda_reparam_kernel<<<blocks, kLambdaThreads, 0, stream>>>(lq1, lk1, lq2, lk2, lambda_init, out,
                                                                      hs, d);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GDA_OK : record_cuda_error(e);
}

}  // namespace gda
