// Instantiations of the fused Q6_K LM-head top-1 kernels for M = 1..17.
#include "launch.cuh"

namespace qgemv {

int launch_lmhead_q6_k(const MmvqArgs& a, int M, cudaStream_t s)
{
    switch (M) {
    case 1: return launch_mmvq_m<FMT_Q6_K, 1, true>(a, s);
    case 2: return launch_mmvq_m<FMT_Q6_K, 2, true>(a, s);
    case 3: return launch_mmvq_m<FMT_Q6_K, 3, true>(a, s);
    case 4: return launch_mmvq_m<FMT_Q6_K, 4, true>(a, s);
    case 5: return launch_mmvq_m<FMT_Q6_K, 5, true>(a, s);
    case 6: return launch_mmvq_m<FMT_Q6_K, 6, true>(a, s);
    case 7: return launch_mmvq_m<FMT_Q6_K, 7, true>(a, s);
    case 8: return launch_mmvq_m<FMT_Q6_K, 8, true>(a, s);
    case 9: return launch_mmvq_m<FMT_Q6_K, 9, true>(a, s);
    case 10: return launch_mmvq_m<FMT_Q6_K, 10, true>(a, s);
    case 11: return launch_mmvq_m<FMT_Q6_K, 11, true>(a, s);
    case 12: return launch_mmvq_m<FMT_Q6_K, 12, true>(a, s);
    case 13: return launch_mmvq_m<FMT_Q6_K, 13, true>(a, s);
    case 14: return launch_mmvq_m<FMT_Q6_K, 14, true>(a, s);
    case 15: return launch_mmvq_m<FMT_Q6_K, 15, true>(a, s);
    case 16: return launch_mmvq_m<FMT_Q6_K, 16, true>(a, s);
    case 17: return launch_mmvq_m<FMT_Q6_K, 17, true>(a, s);
    default: return QGEMV_UNSUPPORTED_SHAPE;
    }
}

unsigned int take_wait_timeouts_lmhead() { return take_wait_timeouts_tu(); }

}  // namespace qgemv
