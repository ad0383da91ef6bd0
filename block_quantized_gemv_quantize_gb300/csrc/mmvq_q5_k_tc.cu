// Host side of the Q5_K x Q8_1 MMVQ (tensor cores, M = 1..17): the plan and
// the launch over the Q5_K pack (one contiguous region per job, no tensor
// maps).
#include "mmvq_tc_host.cuh"

namespace qgemv {

namespace {

// info (when not null): {1, cluster size, grid, ring stages, blocks per job}
// of the plan; nothing is launched.
template <int M>
int launch_q5_k_m(const MmvqArgs& m, cudaStream_t s, int* info)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QGEMV_CUDA_ERROR;
    unsigned int* timeouts = tc_prepare<TCF_Q5_K, M, false>(di, dev);
    if (!timeouts) return QGEMV_CUDA_ERROR;
    TcPlan p{};
    if (!tc_plan<TCF_Q5_K, M, false>(di, dev, m.K, m.N, 0, p)) return QGEMV_UNSUPPORTED_SHAPE;
    if (info) {
        info[0] = 1;
        info[1] = p.C;
        info[2] = p.grid;
        info[3] = p.S;
        info[4] = p.jb;
        return QGEMV_OK;
    }
    CUtensorMap none{};  // the Q5_K kernel reads the pack directly
    TcArgs a{};
    a.xq = m.xq;
    a.y = m.y;
    a.ldy = m.ldy;
    a.w0 = static_cast<const uint8_t*>(m.w_pack);
    a.w1 = a.w0;
    a.K = m.K;
    a.N = m.N;
    a.stages = p.S;
    a.jb = p.jb;
    a.nkb_max = p.nkb_max;
    a.out_tiles = p.out_tiles;
    if (tc_launch<TCF_Q5_K, M, false>(p, a, none, none, none, none, timeouts, s) != cudaSuccess)
        return QGEMV_CUDA_ERROR;
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

}  // namespace

int launch_mmvq_q5_k(const MmvqArgs& a, int M, cudaStream_t s, int* info)
{
    switch (M) {
    case 1: return launch_q5_k_m<1>(a, s, info);
    case 2: return launch_q5_k_m<2>(a, s, info);
    case 3: return launch_q5_k_m<3>(a, s, info);
    case 4: return launch_q5_k_m<4>(a, s, info);
    case 5: return launch_q5_k_m<5>(a, s, info);
    case 6: return launch_q5_k_m<6>(a, s, info);
    case 7: return launch_q5_k_m<7>(a, s, info);
    case 8: return launch_q5_k_m<8>(a, s, info);
    case 9: return launch_q5_k_m<9>(a, s, info);
    case 10: return launch_q5_k_m<10>(a, s, info);
    case 11: return launch_q5_k_m<11>(a, s, info);
    case 12: return launch_q5_k_m<12>(a, s, info);
    case 13: return launch_q5_k_m<13>(a, s, info);
    case 14: return launch_q5_k_m<14>(a, s, info);
    case 15: return launch_q5_k_m<15>(a, s, info);
    case 16: return launch_q5_k_m<16>(a, s, info);
    case 17: return launch_q5_k_m<17>(a, s, info);
    default: return QGEMV_UNSUPPORTED_SHAPE;
    }
}


}  // namespace qgemv
