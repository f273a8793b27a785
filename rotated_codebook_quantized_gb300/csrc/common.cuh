// Shared device helpers of the CUDA library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>
#include <unordered_map>

#include "tq.h"

#define TQ_DEVFN __device__ __forceinline__

namespace tq {

constexpr unsigned kFull = 0xffffffffu;

// fn(integral_constant<int, I>) for I = B .. E-1, expanded at compile time.
template <int B, int E, class Fn>
TQ_DEVFN void static_for(Fn&& fn) {
    if constexpr (B < E) {
        fn(std::integral_constant<int, B>{});
        static_for<B + 1, E>(fn);
    }
}

// ---------------------------------------------------------------- launch helpers

inline tq_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Cycle budget of each bounded wait in the tensor-core kernels launched now (tq_set_wait_budget).
long long wait_budget();

// Programmatic dependent launch.  A kernel launched with launch_pdl may start while the kernel
// before it in the stream is still running: it calls pdl_wait() before it reads or writes any
// memory that kernel may touch (pdl_wait returns once that kernel has completed and its writes
// are visible; launched without the attribute it returns at once), and pdl_trigger() as soon as
// its own successor may be scheduled.  Chained this way each launch's setup overlaps the tail of
// the one before, inside CUDA graphs too.
TQ_DEVFN void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
TQ_DEVFN void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <class... KArgs, class... Args>
inline tq_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

// Raise a kernel's dynamic shared-memory limit once per process (not on every
// launch, so launches can be captured into CUDA graphs without extra API calls).
inline cudaError_t ensure_smem(const void* kernel, size_t bytes) {
    static std::mutex mu;
    static std::unordered_map<const void*, size_t> done;
    if (bytes <= 48 * 1024) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu);
    size_t& cur = done[kernel];
    if (cur >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) cur = bytes;
    return e;
}

inline bool is_pow2(long long v) { return v > 0 && (v & (v - 1)) == 0; }

inline int ilog2(long long v) {
    int r = 0;
    while ((1ll << (r + 1)) <= v) ++r;
    return r;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Codes per word for a codebook size (3 -> 20 trits; 2^b -> 32/b, 3-bit -> 10).
inline int host_codes_per_word(int levels) {
    switch (levels) {
        case 2: return 32;
        case 3: return 20;
        case 4: return 16;
        case 8: return 10;
        case 16: return 8;
        case 256: return 4;
        default: return 0;
    }
}

// ---------------------------------------------------------------- dtype access

TQ_DEVFN float load_as_float(const void* p, int64_t i, int dt) {
    if (dt == TQ_F32) return reinterpret_cast<const float*>(p)[i];
    if (dt == TQ_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
    return __half2float(reinterpret_cast<const __half*>(p)[i]);
}

TQ_DEVFN void store_from_float(void* p, int64_t i, int dt, float v) {
    if (dt == TQ_F32) reinterpret_cast<float*>(p)[i] = v;
    else if (dt == TQ_BF16) reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    else reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
}

TQ_DEVFN float half_bits_to_float(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// ---------------------------------------------------------------- base-3 digits

// Divide-free decode of a trit word w = sum_j d_j 3^j (w < 3^20).
//
// The word is split into two 10-digit halves, hi = w / 3^10 and lo = w mod 3^10
// (a division by a constant, which the compiler turns into a multiply).  Each
// half h < 3^10 becomes a 32-bit fixed-point fraction F = h*72736 + 8860, which
// lies in [h, h+1) * 2^32 / 3^10 for every h (checked exhaustively), so its
// base-3 expansion starts with the ten digits of h.  Each digit then costs one
// 32x32->64-bit multiply-add: (F*3 + 0x4B000000 << 32) puts the next digit d
// in the high word as the float 2^23 + d and the remaining fraction in the low
// word.  Digits come out most significant first.
struct TritHalves {
    uint32_t hi, lo;  // fixed-point fractions of digits 19..10 and 9..0
};

TQ_DEVFN TritHalves trit_split(uint32_t w) {
    uint32_t h = w / 59049u;
    uint32_t l = w - h * 59049u;
    return {h * 72736u + 8860u, l * 72736u + 8860u};
}

// Next digit (most significant first) of a fixed-point fraction, as a float in {0,1,2}.
TQ_DEVFN float trit_next(uint32_t& F) {
    unsigned long long p = (unsigned long long)F * 3ull + (0x4B000000ull << 32);
    F = (uint32_t)p;
    return __uint_as_float((uint32_t)(p >> 32)) - 8388608.0f;
}

// Same digit as an integer.
TQ_DEVFN uint32_t trit_next_int(uint32_t& F) {
    unsigned long long p = (unsigned long long)F * 3ull;
    F = (uint32_t)p;
    return (uint32_t)(p >> 32);
}

// ---------------------------------------------------------------- Walsh-Hadamard transform

// In-place unnormalised fast Walsh-Hadamard transform, block-diagonal with
// blocks of `block` elements, of a vector spread over the CTA: thread t holds
// elements [t*E, t*E+E) in v[].  Stages h = 1, 2, 4, ... < block pair element i
// with i ^ h (the Sylvester order).  Stages inside a thread run in registers,
// stages within a warp use shuffles, the rest go through shared memory `s`
// (at least nthreads*E floats).  All threads of the CTA must call it.
// Floats of shared memory fwht_cta needs for n elements (one pad float per 32).
inline __host__ __device__ constexpr size_t fwht_pad_floats(size_t n) { return n + n / 32; }

template <int E>
TQ_DEVFN void fwht_cta(float (&v)[E], float* s, int block) {  // s: fwht_pad_floats(threads * E) floats
    const int lane = threadIdx.x & 31;
    int h = 1;
#pragma unroll
    for (int hh = 1; hh < E; hh <<= 1) {
        if (hh < block) {
#pragma unroll
            for (int i = 0; i < E; ++i) {
                if (!(i & hh)) {
                    float a = v[i], b = v[i + hh];
                    v[i] = a + b;
                    v[i + hh] = a - b;
                }
            }
        }
    }
    h = E;
    for (; h < block && h < 32 * E; h <<= 1) {
        const int m = h / E;
        // the upper lane of a pair keeps o - v, the lower v + o: one fma with a sign of +-1 (exact)
        const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const float o = __shfl_xor_sync(kFull, v[i], m);
            v[i] = fmaf(sgn, v[i], o);
        }
    }
    if (h < block) {
        // Element i sits at i + i / 32: a thread's E consecutive elements would otherwise put
        // the lanes of one access E floats apart, an E-way bank conflict (fwht_pad_floats).
        const int base = threadIdx.x * E;
        for (; h < block; h <<= 1) {
#pragma unroll
            for (int i = 0; i < E; ++i) s[(base + i) + ((base + i) >> 5)] = v[i];
            __syncthreads();
            const float sgn = (base & h) ? -1.0f : 1.0f;  // h >= 32 E: the same side for all of the thread's E
#pragma unroll
            for (int i = 0; i < E; ++i) {
                const int j = (base + i) ^ h;
                v[i] = fmaf(sgn, v[i], s[j + (j >> 5)]);
            }
            __syncthreads();
        }
    }
}

// Unnormalised FWHT of 128 values held 4 per lane by one warp (lane l holds
// elements 4l..4l+3).
TQ_DEVFN void fwht_warp128(float (&v)[4]) {
    const int lane = threadIdx.x & 31;
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[2] = a0 - a2;
    v[1] = a1 + a3;
    v[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        // the upper lane of a pair keeps o - v, the lower v + o: one fma with a sign of +-1 (exact)
        const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(kFull, v[i], m);
            v[i] = fmaf(sgn, v[i], o);
        }
    }
}

}  // namespace tq
