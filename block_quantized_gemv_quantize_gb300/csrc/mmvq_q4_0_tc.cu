// Host side of the tensor-core Q4_0 MMVQ: tensor maps over the packed
// weight, the launch plan (cluster size, ring depth) and the launch, for
// M = 1..17, one weight or a pair.
#include <atomic>

#include "mmvq_tc_host.cuh"

namespace qgemv {

namespace {

std::atomic<int> g_tc_enabled{1};

// info (when not null): {1, cluster size, grid, ring stages} of the plan.
template <int M, bool PAIR>
int launch_tc_m(const MmvqArgs& m, cudaStream_t s, int* info)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QGEMV_CUDA_ERROR;
    unsigned int* timeouts = tc_prepare<TCF_Q4_0, M, PAIR>(di, dev);
    if (!timeouts) return QGEMV_CUDA_ERROR;
    TcPlan p{};
    if (!tc_plan<TCF_Q4_0, M, PAIR>(di, dev, m.K, m.N, PAIR ? m.N2 : 0, p)) return TC_NOT_TAKEN;
    if (info) {
        info[0] = 1;
        info[1] = p.C;
        info[2] = p.grid;
        info[3] = p.S;
        return QGEMV_OK;
    }
    CUtensorMap n0, d0, n1, d1;
    if (!q4_0_tensor_maps(m.w_pack, m.N, m.K, p.jb, &n0, &d0)) return QGEMV_CUDA_ERROR;
    if (PAIR) {
        if (!q4_0_tensor_maps(m.w_pack2, m.N2, m.K, p.jb, &n1, &d1)) return QGEMV_CUDA_ERROR;
    } else {
        n1 = n0;
        d1 = d0;
    }
    TcArgs a{};
    a.xq = m.xq;
    a.y = m.y;
    a.y2 = PAIR ? m.y2 : nullptr;
    a.ldy = m.ldy;
    a.res = PAIR ? nullptr : m.x;  // a residual call passes the residual in the activation field
    a.ldr = m.ldx;
    a.K = m.K;
    a.N = m.N;
    a.N2 = PAIR ? m.N2 : 0;
    a.stages = p.S;
    a.jb = p.jb;
    a.nkb_max = p.nkb_max;
    a.out_tiles = p.out_tiles;
    if (tc_launch<TCF_Q4_0, M, PAIR>(p, a, n0, d0, n1, d1, timeouts, s) != cudaSuccess) return QGEMV_CUDA_ERROR;
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

template <bool PAIR>
int launch_tc(const MmvqArgs& a, int M, cudaStream_t s, int* info)
{
    switch (M) {
    case 1: return launch_tc_m<1, PAIR>(a, s, info);
    case 2: return launch_tc_m<2, PAIR>(a, s, info);
    case 3: return launch_tc_m<3, PAIR>(a, s, info);
    case 4: return launch_tc_m<4, PAIR>(a, s, info);
    case 5: return launch_tc_m<5, PAIR>(a, s, info);
    case 6: return launch_tc_m<6, PAIR>(a, s, info);
    case 7: return launch_tc_m<7, PAIR>(a, s, info);
    case 8: return launch_tc_m<8, PAIR>(a, s, info);
    case 9: return launch_tc_m<9, PAIR>(a, s, info);
    case 10: return launch_tc_m<10, PAIR>(a, s, info);
    case 11: return launch_tc_m<11, PAIR>(a, s, info);
    case 12: return launch_tc_m<12, PAIR>(a, s, info);
    case 13: return launch_tc_m<13, PAIR>(a, s, info);
    case 14: return launch_tc_m<14, PAIR>(a, s, info);
    case 15: return launch_tc_m<15, PAIR>(a, s, info);
    case 16: return launch_tc_m<16, PAIR>(a, s, info);
    case 17: return launch_tc_m<17, PAIR>(a, s, info);
    default: return TC_NOT_TAKEN;
    }
}

}  // namespace

int set_q4_0_tensor_cores(int mode) { return g_tc_enabled.exchange(mode >= 0 && mode <= 2 ? mode : 1); }

int launch_mmvq_q4_0_tc(const MmvqArgs& a, int M, bool pair, cudaStream_t s, int* info)
{
    const int mode = g_tc_enabled.load();
    if (!mode) return TC_NOT_TAKEN;
    if (a.N % TC_ROWS || (pair && a.N2 % TC_ROWS) || a.K % (CHUNK * QK)) return TC_NOT_TAKEN;
    // Below 5 rows the SIMT kernels are as fast or faster on the verifier's
    // weights (their fixed cost per call is lower: 1-2 us better at N = 5120
    // and 17408, K = 5120), but on large weights the small-M kernel streams
    // faster at any M (N = 248320, K = 5120, M = 1..4: 109-113 us against
    // 115-120 us on dp4a, back to back).
    if (M < TC_MIN_M) {
        const int64_t elems = (int64_t)(a.N + (pair ? a.N2 : 0)) * a.K;
        if (mode != 1 || elems < TC_SMALL_M_MIN_ELEMS) return TC_NOT_TAKEN;
        return launch_mmvq_q4_0_mma(a, M, pair, s, info);  // TC_NOT_TAKEN without a plan
    }
    if (mode == 1 && M <= 8) {  // one 8-column MMA tile: the small-M kernel, where it has a plan
        const int st = launch_mmvq_q4_0_mma(a, M, pair, s, info);
        if (st != TC_NOT_TAKEN) return st;
    }
    return pair ? launch_tc<true>(a, M, s, info) : launch_tc<false>(a, M, s, info);
}


}  // namespace qgemv
