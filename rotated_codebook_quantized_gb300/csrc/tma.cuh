// mbarrier, tensor-copy (TMA) and async-proxy helpers shared by the staged
// kernels, and the host lookup of the driver's tensor-map encoder.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"

namespace tq {

constexpr long long kWaitCycles = 1ll << 31;  // about a second at GB300 clocks

TQ_DEVFN uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

TQ_DEVFN void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

TQ_DEVFN void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

// The waiting thread is suspended (issuing nothing) until the phase completes
// or about kSuspendNs elapse, so idle roles leave the issue slots to the others.
constexpr uint32_t kSuspendNs = 20000;
TQ_DEVFN bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Wait bounded by time only (used to drain copies or MMAs still in flight).
TQ_DEVFN bool mbar_wait_drain(uint64_t* b, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// Has the phase of parity `parity` completed?  (try_wait without a time hint: when the phase
// is not complete the thread may still be held for a system-dependent time; mbar_peek never is.)
TQ_DEVFN bool mbar_test(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the phase (mbarrier.test_wait never suspends the thread, unlike
// try_wait, which may wait for the phase up to a system-dependent time).
TQ_DEVFN bool mbar_peek(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.  Returns false
// (and raises the CTA's abort flag) if it did not within `budget` cycles
// (kWaitCycles unless the launch carries another budget) or if another role
// already aborted.
TQ_DEVFN bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag, long long budget = kWaitCycles) {
    if (mbar_test(b, parity)) return true;  // common case first: no clock read, no suspension
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > budget) {
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// The same bounded wait, polling with short sleeps (for waits expected to be brief, where a
// long suspension would outlast the event).
TQ_DEVFN bool mbar_wait_short(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                               long long budget = kWaitCycles) {
    if (mbar_test(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_test(b, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > budget) {
            *abort_flag = 1;
            return false;
        }
        __nanosleep(32);
    }
    return true;
}

TQ_DEVFN void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Makes barrier initialisation visible to the async proxy (tensor copies).
TQ_DEVFN void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

TQ_DEVFN void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
TQ_DEVFN void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
TQ_DEVFN void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

// The driver's tensor-map encoder, looked up once through the runtime (no link
// against the driver library); null if the driver does not provide it.
inline EncodeFn tensor_map_encoder() {
    static const EncodeFn fn = []() -> EncodeFn {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeFn>(f);
    }();
    return fn;
}

}  // namespace tq
