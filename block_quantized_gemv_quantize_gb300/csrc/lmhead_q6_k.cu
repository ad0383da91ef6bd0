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

namespace {

template <int M>
int lmhead_plan_m(int K, int N, int* info)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    const MmvqPlan p = mmvq_plan<FMT_Q6_K, M, true>(di, K, N);
    info[0] = p.ring ? 1 : 0;
    info[1] = p.grid;
    info[2] = p.warps;
    info[3] = p.ring ? p.stages : 0;
    return QGEMV_OK;
}

}  // namespace

int lmhead_q6_k_plan(int M, int K, int N, int* info)
{
    switch (M) {
    case 1: return lmhead_plan_m<1>(K, N, info);
    case 2: return lmhead_plan_m<2>(K, N, info);
    case 3: return lmhead_plan_m<3>(K, N, info);
    case 4: return lmhead_plan_m<4>(K, N, info);
    case 5: return lmhead_plan_m<5>(K, N, info);
    case 6: return lmhead_plan_m<6>(K, N, info);
    case 7: return lmhead_plan_m<7>(K, N, info);
    case 8: return lmhead_plan_m<8>(K, N, info);
    case 9: return lmhead_plan_m<9>(K, N, info);
    case 10: return lmhead_plan_m<10>(K, N, info);
    case 11: return lmhead_plan_m<11>(K, N, info);
    case 12: return lmhead_plan_m<12>(K, N, info);
    case 13: return lmhead_plan_m<13>(K, N, info);
    case 14: return lmhead_plan_m<14>(K, N, info);
    case 15: return lmhead_plan_m<15>(K, N, info);
    case 16: return lmhead_plan_m<16>(K, N, info);
    case 17: return lmhead_plan_m<17>(K, N, info);
    default: return QGEMV_UNSUPPORTED_SHAPE;
    }
}


}  // namespace qgemv
