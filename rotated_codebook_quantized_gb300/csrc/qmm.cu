// Placeholder translation unit for the expert-sorted gather-GEMM (tcgen05).
#include "common.cuh"

extern "C" size_t tq_gather_qmm_workspace_bytes(int32_t experts) { return experts > 0 ? 256 : 0; }

extern "C" tq_status tq_gather_qmm(const tq_qweight_t* w, const void* x, tq_dtype xdt, const int32_t* perm,
                                   const int32_t* offsets, int32_t P, int32_t k, int32_t per_pair_input, void* y,
                                   tq_dtype ydt, void* ws, size_t ws_bytes, uint32_t* err, void* stream) {
    return TQ_ERR_UNSUPPORTED;
}
