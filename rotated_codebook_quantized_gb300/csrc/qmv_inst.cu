// One (levels, group) instantiation of the inline-decode matvec.  The build
// compiles this file once per pair with -DTQ_LEVELS=<L> -DTQ_GROUP=<G>, so the
// instantiations compile in parallel.
#include "qmv_impl.cuh"

#if !defined(TQ_LEVELS) || !defined(TQ_GROUP)
#error "compile with -DTQ_LEVELS and -DTQ_GROUP"
#endif

#define TQ_CAT_(a, b, c) a##b##_g##c
#define TQ_CAT(a, b, c) TQ_CAT_(a, b, c)

namespace tq {
tq_status TQ_CAT(qmv_run_l, TQ_LEVELS, TQ_GROUP)(QmvParams p, int nv, int n_items, cudaStream_t st) {
    return dispatch_qmv_nv<TQ_LEVELS, TQ_GROUP>(p, nv, n_items, st);
}
}  // namespace tq
