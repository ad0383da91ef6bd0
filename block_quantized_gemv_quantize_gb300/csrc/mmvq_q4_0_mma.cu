// The small-M tensor-core Q4_0 MMVQ for one weight (the pair form is in
// mmvq_q4_0_mma_pair.cu), and the entry that picks between them.
#include "mmvq_q4_0_mma_host.cuh"

namespace qgemv {

int launch_mmvq_q4_0_mma_pair(const MmvqArgs& a, int M, cudaStream_t s, int* info);

int launch_mmvq_q4_0_mma(const MmvqArgs& a, int M, bool pair, cudaStream_t s, int* info)
{
    return pair ? launch_mmvq_q4_0_mma_pair(a, M, s, info) : launch_qm<false>(a, M, s, info);
}


}  // namespace qgemv
