// Instantiations of the Q4_0 x Q8_1 MMVQ kernels for M = 1..17.
#include "launch.cuh"

namespace qgemv {

int launch_mmvq_q4_0(const MmvqArgs& a, int M, cudaStream_t s)
{
    switch (M) {
    case 1: return launch_mmvq_m<FMT_Q4_0, 1, false>(a, s);
    case 2: return launch_mmvq_m<FMT_Q4_0, 2, false>(a, s);
    case 3: return launch_mmvq_m<FMT_Q4_0, 3, false>(a, s);
    case 4: return launch_mmvq_m<FMT_Q4_0, 4, false>(a, s);
    case 5: return launch_mmvq_m<FMT_Q4_0, 5, false>(a, s);
    case 6: return launch_mmvq_m<FMT_Q4_0, 6, false>(a, s);
    case 7: return launch_mmvq_m<FMT_Q4_0, 7, false>(a, s);
    case 8: return launch_mmvq_m<FMT_Q4_0, 8, false>(a, s);
    case 9: return launch_mmvq_m<FMT_Q4_0, 9, false>(a, s);
    case 10: return launch_mmvq_m<FMT_Q4_0, 10, false>(a, s);
    case 11: return launch_mmvq_m<FMT_Q4_0, 11, false>(a, s);
    case 12: return launch_mmvq_m<FMT_Q4_0, 12, false>(a, s);
    case 13: return launch_mmvq_m<FMT_Q4_0, 13, false>(a, s);
    case 14: return launch_mmvq_m<FMT_Q4_0, 14, false>(a, s);
    case 15: return launch_mmvq_m<FMT_Q4_0, 15, false>(a, s);
    case 16: return launch_mmvq_m<FMT_Q4_0, 16, false>(a, s);
    case 17: return launch_mmvq_m<FMT_Q4_0, 17, false>(a, s);
    default: return QGEMV_UNSUPPORTED_SHAPE;
    }
}


}  // namespace qgemv
