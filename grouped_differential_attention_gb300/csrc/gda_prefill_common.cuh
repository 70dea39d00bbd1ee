// Pieces shared by the two tensor-core prefill kernels: cluster and mbarrier
// helpers, and the QK / PV MMA issue sequences for 128-row query tiles.
#pragma once

#include <cstdint>

#include "gda.h"
#include "gda_device.cuh"

namespace gda {
namespace {

constexpr int kBM = 128;          // query rows per CTA (= TMEM lanes)
constexpr int kDVS = 128;         // dv columns per CTA

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Shared-memory address of `local`'s counterpart in CTA `peer` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void *local, uint32_t peer) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(peer));
    return remote;
}

__device__ __forceinline__ void st_cluster_f32(const float *local, uint32_t peer, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr(local, peer)), "f"(v) : "memory");
}

// Wait used while winding down: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, unsigned *err) {
    int dummy = 0;
    mbar_wait(bar, parity, err, GDA_DEVERR_PREFILL_TIMEOUT, &dummy);
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, unsigned *err,
                                         volatile int *abort) {
    return mbar_wait(bar, parity, err, GDA_DEVERR_PREFILL_TIMEOUT, abort);
}

// Whole-warp wait: every lane polls, the result is agreed by vote so the
// warp stays converged for the .sync.aligned tcgen05 instructions after it.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, unsigned *err,
                                          volatile int *abort) {
    bool ok = wait_bar(bar, parity, err, abort);
    return __all_sync(0xffffffffu, ok);
}

// S = Q K^T for a 128-row query tile and BN keys: K-major operands with the
// 128-byte swizzle (64-element column blocks, 8-row groups 1 KiB apart).
template <int D, int BN>
__device__ __forceinline__ void issue_qk(uint32_t tS, uint32_t qa, uint32_t ka) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, 0);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        const uint32_t blk = k / 4, sub = (k % 4) * 32;
        const uint64_t a = smem_desc_sw128(qa + blk * (kBM * 128) + sub, 16, 1024);
        const uint64_t b = smem_desc_sw128(ka + blk * (BN * 128) + sub, 16, 1024);
        mma_ss(tS, a, b, idesc, k > 0 ? 1u : 0u);
    }
}

// O += P V with P (bf16 pairs, BN keys) in TMEM columns tP .. tP + BN/2 and
// the V stage as an MN-major B operand: two [BN x 64] column blocks, rows of
// 128 B, 128-byte swizzle; 8-row K groups 1024 B apart, N blocks BN*128 B apart.
template <int BN>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint32_t va, bool acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kDVS, 1);
#pragma unroll
    for (int k = 0; k < BN / 16; ++k) {
        const uint64_t b = smem_desc_sw128(va + k * 2048, BN * 128, 1024);
        mma_ts(tO, tP + k * 8, b, idesc, (acc || k > 0) ? 1u : 0u);
    }
}

// OR of `pred` over the `count` threads that reach named barrier `id`.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return out != 0;
}

// Arrive on the peer CTA's mbarrier (release at cluster scope: the data
// stored to the peer before this arrive is visible to its waiter).
__device__ __forceinline__ void mbar_arrive_remote(uint64_t *local_bar, uint32_t peer) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr(local_bar, peer))
                 : "memory");
}

// Bounded wait with acquire at cluster scope (pairs with mbar_arrive_remote).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, unsigned *err,
                                                  volatile int *abort) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((it & 15u) == 15u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                atomicOr(err, GDA_DEVERR_PREFILL_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

}  // namespace
}  // namespace gda
