// Row-wise randomized Hadamard rotation: tq_rotate and tq_swiglu_rotate.
//
// "How it works", "Running a quantized layer": the layer rotates its input,
// x_rot = R x with R = blockdiag(H_b) diag(signs) / sqrt(b).  One CTA per span
// of whole blocks of a row; each thread holds E consecutive elements, the
// transform runs in registers, warp shuffles and shared memory (fwht_cta).
#include <math.h>

#include "common.cuh"

using namespace tq;

namespace {

struct PlainLoad {
    const void* x;
    int dt;
    TQ_DEVFN float operator()(int64_t row, int dim, int i) const { return load_as_float(x, row * dim + i, dt); }
};

// silu(gate) * up for one element of a [P, 2*inter] gate||up row.
struct SwigluLoad {
    const float* gu;
    TQ_DEVFN float operator()(int64_t row, int dim, int i) const {
        const float g = gu[row * 2 * dim + i];
        const float u = gu[row * 2 * dim + dim + i];
        return g / (1.0f + expf(-g)) * u;
    }
};

// One CTA per span of a row (span = a whole number of Hadamard blocks, so
// CTAs are independent); thread t holds elements t*E .. t*E+E-1 of the span.
template <int E, class Load>
__global__ void __launch_bounds__(1024) rotate_rows_kernel(Load ld, int dim, int span, int block, float scale,
                                                           const int8_t* __restrict__ signs, void* out, int odt) {
    extern __shared__ float s[];
    pdl_trigger();
    pdl_wait();
    const int spans = dim / span;
    const int64_t row = blockIdx.x / spans;
    const int base = (blockIdx.x - (int)(row * spans)) * span + threadIdx.x * E;
    int8_t sg[E];
    bool done = false;
    if constexpr (E >= 4) {  // E consecutive signs in 4-byte words when the table is 4-byte aligned
        if ((reinterpret_cast<uintptr_t>(signs) & 3) == 0) {
#pragma unroll
            for (int i = 0; i < E; i += 4) {
                const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(signs + base + i));
#pragma unroll
                for (int b = 0; b < 4; ++b) sg[i + b] = (int8_t)(w >> (8 * b));
            }
            done = true;
        }
    }
    if (!done) {
#pragma unroll
        for (int i = 0; i < E; ++i) sg[i] = signs[base + i];
    }
    float v[E];
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = ld(row, dim, base + i) * (float)sg[i];
    fwht_cta<E>(v, s, block);
#pragma unroll
    for (int i = 0; i < E; ++i) store_from_float(out, row * dim + base + i, odt, v[i] * scale);
}

// Span: block times the largest power of two m with block * m <= 2048 and
// dim % (block * m) == 0 (a block above 2048 is its own span).  Elements per
// thread: span / 512 (at least 1, at most 16): up to 512 threads keep many
// loads in flight, and span / E <= 1024 threads in whole warps.
int pick_span(int dim, int block) {
    int span = block;
    while (span * 2 <= 2048 && dim % (span * 2) == 0) span *= 2;
    return span;
}
int pick_e(int span) {
    int e = span / 512;
    if (e < 1) e = 1;
    if (e > 16) e = 16;
    while (e > 1 && span % (32 * e) != 0) e >>= 1;
    return (span % (32 * e) == 0 && span / e <= 1024) ? e : 0;
}

bool rotation_ok(const tq_rotation_t* rot) {
    return rot && rot->signs && rot->dim > 0 && is_pow2(rot->block) && rot->block <= 8192 &&
           rot->dim % rot->block == 0;
}

template <class Load>
tq_status launch_rotate(const Load& ld, int64_t rows, const tq_rotation_t* rot, void* out, tq_dtype odt,
                        cudaStream_t st) {
    const int dim = rot->dim, block = rot->block;
    const int span = pick_span(dim, block);
    const int e = pick_e(span);
    if (e == 0) return TQ_ERR_UNSUPPORTED;
    if (rows == 0) return TQ_OK;
    if (rows * (dim / span) > 0x7fffffffll) return TQ_ERR_INVALID;
    const int threads = span / e;
    const size_t smem = fwht_pad_floats(span) * sizeof(float);
    const float scale = (float)(1.0 / sqrt((double)block));
    const dim3 grid((unsigned)(rows * (dim / span)));
    switch (e) {
#define TQ_ROT_CASE(EE)                                                                                   \
    case EE:                                                                                              \
        if (ensure_smem((const void*)rotate_rows_kernel<EE, Load>, smem) != cudaSuccess) return TQ_ERR_CUDA; \
        return launch_pdl(rotate_rows_kernel<EE, Load>, grid, dim3(threads), smem, st, ld, dim, span, block, scale, \
                          rot->signs, out, (int)odt);
        TQ_ROT_CASE(1)
        TQ_ROT_CASE(2)
        TQ_ROT_CASE(4)
        TQ_ROT_CASE(8)
        TQ_ROT_CASE(16)
#undef TQ_ROT_CASE
        default: return TQ_ERR_UNSUPPORTED;
    }
    return launch_status();
}

bool dtype_ok(int dt) { return dt == TQ_F32 || dt == TQ_BF16 || dt == TQ_F16; }

}  // namespace

extern "C" tq_status tq_rotate(const tq_rotation_t* rot, const void* x, tq_dtype xdt, int64_t rows, void* x_rot,
                               tq_dtype ydt, void* stream) {
    if (!rotation_ok(rot) || rows < 0 || !dtype_ok(xdt) || !dtype_ok(ydt)) return TQ_ERR_INVALID;
    if (rows > 0 && (!x || !x_rot || x == x_rot)) return TQ_ERR_INVALID;
    return launch_rotate(PlainLoad{x, (int)xdt}, rows, rot, x_rot, ydt, as_stream(stream));
}

extern "C" tq_status tq_swiglu_rotate(const float* gate_up, int64_t P, int32_t inter, const tq_rotation_t* rot,
                                      void* h_rot, tq_dtype ydt, void* stream) {
    if (!rotation_ok(rot) || rot->dim != inter || P < 0 || !dtype_ok(ydt)) return TQ_ERR_INVALID;
    if (P > 0 && (!gate_up || !h_rot)) return TQ_ERR_INVALID;
    return launch_rotate(SwigluLoad{gate_up}, P, rot, h_rot, ydt, as_stream(stream));
}
