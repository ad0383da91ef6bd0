// The small-M tensor-core Q4_0 MMVQ for a pair of weights of one K against
// one activation (the verifier's gate and up projections).
#include "mmvq_q4_0_mma_host.cuh"

namespace qgemv {

int launch_mmvq_q4_0_mma_pair(const MmvqArgs& a, int M, cudaStream_t s, int* info)
{
    return launch_qm<true>(a, M, s, info);
}


}  // namespace qgemv
