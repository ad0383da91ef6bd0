// Instantiations of the Q6_K x Q8_1 MMVQ kernels for M = 1..17.
#include "launch.cuh"

namespace qgemv {

int launch_mmvq_q6_k(const MmvqArgs& a, int M, cudaStream_t s)
{
    switch (M) {
    case 1: return launch_mmvq_m<FMT_Q6_K, 1, false>(a, s);
    case 2: return launch_mmvq_m<FMT_Q6_K, 2, false>(a, s);
    case 3: return launch_mmvq_m<FMT_Q6_K, 3, false>(a, s);
    case 4: return launch_mmvq_m<FMT_Q6_K, 4, false>(a, s);
    case 5: return launch_mmvq_m<FMT_Q6_K, 5, false>(a, s);
    case 6: return launch_mmvq_m<FMT_Q6_K, 6, false>(a, s);
    case 7: return launch_mmvq_m<FMT_Q6_K, 7, false>(a, s);
    case 8: return launch_mmvq_m<FMT_Q6_K, 8, false>(a, s);
    case 9: return launch_mmvq_m<FMT_Q6_K, 9, false>(a, s);
    case 10: return launch_mmvq_m<FMT_Q6_K, 10, false>(a, s);
    case 11: return launch_mmvq_m<FMT_Q6_K, 11, false>(a, s);
    case 12: return launch_mmvq_m<FMT_Q6_K, 12, false>(a, s);
    case 13: return launch_mmvq_m<FMT_Q6_K, 13, false>(a, s);
    case 14: return launch_mmvq_m<FMT_Q6_K, 14, false>(a, s);
    case 15: return launch_mmvq_m<FMT_Q6_K, 15, false>(a, s);
    case 16: return launch_mmvq_m<FMT_Q6_K, 16, false>(a, s);
    case 17: return launch_mmvq_m<FMT_Q6_K, 17, false>(a, s);
    default: return QGEMV_UNSUPPORTED_SHAPE;
    }
}


}  // namespace qgemv
