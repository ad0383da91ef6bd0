// Instantiations of the fused Q6_K LM-head top-k kernels for M = 1..17.
#include "launch.cuh"

namespace qgemv {

namespace {

template <int M>
int launch_topk_m(const MmvqArgs& a, cudaStream_t s)
{
    return launch_mmvq_pm<FMT_Q6_K, M, true, false, false, true>(a, s);
}

}  // namespace

int launch_lmhead_q6_k_topk(const MmvqArgs& a, int M, cudaStream_t s)
{
    switch (M) {
    case 1: return launch_topk_m<1>(a, s);
    case 2: return launch_topk_m<2>(a, s);
    case 3: return launch_topk_m<3>(a, s);
    case 4: return launch_topk_m<4>(a, s);
    case 5: return launch_topk_m<5>(a, s);
    case 6: return launch_topk_m<6>(a, s);
    case 7: return launch_topk_m<7>(a, s);
    case 8: return launch_topk_m<8>(a, s);
    case 9: return launch_topk_m<9>(a, s);
    case 10: return launch_topk_m<10>(a, s);
    case 11: return launch_topk_m<11>(a, s);
    case 12: return launch_topk_m<12>(a, s);
    case 13: return launch_topk_m<13>(a, s);
    case 14: return launch_topk_m<14>(a, s);
    case 15: return launch_topk_m<15>(a, s);
    case 16: return launch_topk_m<16>(a, s);
    case 17: return launch_topk_m<17>(a, s);
    default: return QGEMV_UNSUPPORTED_SHAPE;
    }
}

}  // namespace qgemv
