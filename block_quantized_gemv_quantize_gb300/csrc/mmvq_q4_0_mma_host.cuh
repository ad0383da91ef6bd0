// Host side of the small-M tensor-core Q4_0 MMVQ (M = 1..8): the launch
// plan (job shape, cluster size, ring depth), the per-device opt-in and the
// launch.  Included by one translation unit for one weight and one for the
// pair, which compile in parallel.
#pragma once

#include <mutex>

#include "mmvq_q4_0_mma.cuh"
#include "mmvq_tc_host.cuh"

namespace qgemv {
namespace {

// The job shapes: TL tiles of 16 rows x JB blocks.
constexpr int QM_SHAPES = 3;
constexpr int QM_TL[QM_SHAPES] = {2, 1, 1};
constexpr int QM_JB[QM_SHAPES] = {8, 16, 8};

struct QmPlan {
    int C, grid, S, shape, nkb_max, out_units;
    size_t smem;
};

template <int M, int JB, int TL, bool PAIR>
cudaError_t qm_launch(const QmPlan& p, const TcArgs& a, const CUtensorMap& n0, const CUtensorMap& d0,
                      const CUtensorMap& n1, const CUtensorMap& d1, unsigned int* timeouts, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(QM_THREADS);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int na = 1;
    if (p.C > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = p.C;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, mmvq_q4_0_mma_kernel<M, JB, TL, PAIR>, a, n0, d0, n1, d1, timeouts);
}

template <int M, int JB, int TL, bool PAIR>
bool qm_opt_in(int smem)
{
    return cudaFuncSetAttribute(mmvq_q4_0_mma_kernel<M, JB, TL, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem) == cudaSuccess;
}

// Clusters of C CTAs of the kernel that can be resident at once (at the full
// shared memory, which every plan with C > 1 comes close to).
template <int M, int JB, int TL, bool PAIR>
int qm_resident_clusters(int C, int smem)
{
    if (C == 1) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(QM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mmvq_q4_0_mma_kernel<M, JB, TL, PAIR>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    return n;
}

// Per device: every job shape opted in to the full shared memory, the
// timeout counter's address, the resident clusters of each shape and size.
struct QmDevice {
    bool ok;
    unsigned int* timeouts;
    int clusters[QM_SHAPES][4];
};

template <int M, bool PAIR>
const QmDevice& qm_device(const DeviceInfo& di, int dev)
{
    static QmDevice d[64];
    static std::once_flag once[64];
    std::call_once(once[dev], [&]() {
        QmDevice& q = d[dev];
        const int sm = di.smem_optin;
        q.ok = qm_opt_in<M, QM_JB[0], QM_TL[0], PAIR>(sm) && qm_opt_in<M, QM_JB[1], QM_TL[1], PAIR>(sm) &&
               qm_opt_in<M, QM_JB[2], QM_TL[2], PAIR>(sm) &&
               (q.timeouts = wait_timeout_counter()) != nullptr;
        for (int ci = 0; ci < 4; ++ci) {
            const int C = TC_CLUSTERS[ci];
            int r[QM_SHAPES] = {0, 0, 0};
            if (q.ok) {
                r[0] = qm_resident_clusters<M, QM_JB[0], QM_TL[0], PAIR>(C, sm);
                r[1] = qm_resident_clusters<M, QM_JB[1], QM_TL[1], PAIR>(C, sm);
                r[2] = qm_resident_clusters<M, QM_JB[2], QM_TL[2], PAIR>(C, sm);
            }
            for (int k = 0; k < QM_SHAPES; ++k) q.clusters[k][ci] = C == 1 ? di.sms : r[k];
        }
        if (!q.ok) cudaGetLastError();
    });
    return d[dev];
}

// The cheapest plan over job shapes and cluster sizes (1, 2, 4, 8): the
// critical warp's jobs times a job's cost in 16-row x 8-block units (a
// two-tile job costs 1.6 of them: it shares the activation loads; a 16-block
// job 1.9: it halves the per-job copy and loop overhead), plus two units for
// the cross-CTA combine when C > 1.  A plan needs at least two ring stages
// next to the activation and the cluster's combine area, and at most
// QM_UNITS activation units per thread; false when none fits (the general
// tensor-core kernel then takes the shape).
template <int M, bool PAIR>
bool qm_plan(const DeviceInfo& di, const QmDevice& qd, int K, int N, int N2, QmPlan& best)
{
    const int NB = K / QK;
    bool found = false;
    double best_cost = 0.0;
    for (int k = 0; k < QM_SHAPES; ++k) {
        const int TL = QM_TL[k], jb = QM_JB[k];
        if (NB % jb) continue;
        const int64_t T = (N / TC_ROWS + TL - 1) / TL + (PAIR ? (N2 / TC_ROWS + TL - 1) / TL : 0);
        const int njb = NB / jb;
        for (int ci = 0; ci < 4; ++ci) {
            const int C = TC_CLUSTERS[ci];
            if (njb < C) break;
            const int jpt = (njb + C - 1) / C;
            const int nkb = jpt * jb;
            if (nkb * M > QM_UNITS * QM_THREADS) continue;
            int64_t ncl = qd.clusters[k][ci];
            if (ncl <= 0) continue;
            if (ncl > T) ncl = T;
            const int units = (int)((T + ncl - 1) / ncl);
            const int out_units = C > 1 ? units : 0;
            int S = 0;
            for (int s = QM_MAX_STAGES; s >= 2 && S == 0; --s)
                if (qm_smem(M, s, jb, TL, nkb, out_units).bytes <= (uint32_t)di.smem_optin) S = s;
            if (S == 0) continue;
            const double unit = TL == 2 ? 1.6 : jb == 16 ? 1.9 : 1.0;
            const double cost =
                (double)(((int64_t)units * jpt + QM_WARPS - 1) / QM_WARPS) * unit + (C > 1 ? 2.0 : 0.0);
            if (!found || cost < best_cost - 1e-9) {
                found = true;
                best_cost = cost;
                best.C = C;
                best.grid = (int)(ncl * C);
                best.S = S;
                best.shape = k;
                best.nkb_max = nkb;
                best.out_units = out_units;
                best.smem = qm_smem(M, S, jb, TL, nkb, out_units).bytes;
            }
        }
    }
    return found;
}

template <int M, bool PAIR>
int launch_qm_m(const MmvqArgs& m, cudaStream_t s, int* info)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QGEMV_CUDA_ERROR;
    const QmDevice& qd = qm_device<M, PAIR>(di, dev);
    if (!qd.ok) return QGEMV_CUDA_ERROR;
    QmPlan p{};
    if (!qm_plan<M, PAIR>(di, qd, m.K, m.N, PAIR ? m.N2 : 0, p)) return TC_NOT_TAKEN;
    if (info) {
        info[0] = 2;
        info[1] = p.C;
        info[2] = p.grid;
        info[3] = p.S;
        return QGEMV_OK;
    }
    const int TL = QM_TL[p.shape], jb = QM_JB[p.shape];
    CUtensorMap n0, d0, n1, d1;
    if (!q4_0_tensor_maps(m.w_pack, m.N, m.K, jb, &n0, &d0, TL)) return QGEMV_CUDA_ERROR;
    if (PAIR) {
        if (!q4_0_tensor_maps(m.w_pack2, m.N2, m.K, jb, &n1, &d1, TL)) return QGEMV_CUDA_ERROR;
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
    a.jb = jb;
    a.nkb_max = p.nkb_max;
    a.out_tiles = p.out_units;
    a.drop_copy = take_drop_request();
    cudaError_t e;
    switch (p.shape) {
    case 0: e = qm_launch<M, QM_JB[0], QM_TL[0], PAIR>(p, a, n0, d0, n1, d1, qd.timeouts, s); break;
    case 1: e = qm_launch<M, QM_JB[1], QM_TL[1], PAIR>(p, a, n0, d0, n1, d1, qd.timeouts, s); break;
    default: e = qm_launch<M, QM_JB[2], QM_TL[2], PAIR>(p, a, n0, d0, n1, d1, qd.timeouts, s); break;
    }
    if (e != cudaSuccess) return QGEMV_CUDA_ERROR;
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

template <bool PAIR>
int launch_qm(const MmvqArgs& a, int M, cudaStream_t s, int* info)
{
    switch (M) {
    case 1: return launch_qm_m<1, PAIR>(a, s, info);
    case 2: return launch_qm_m<2, PAIR>(a, s, info);
    case 3: return launch_qm_m<3, PAIR>(a, s, info);
    case 4: return launch_qm_m<4, PAIR>(a, s, info);
    case 5: return launch_qm_m<5, PAIR>(a, s, info);
    case 6: return launch_qm_m<6, PAIR>(a, s, info);
    case 7: return launch_qm_m<7, PAIR>(a, s, info);
    case 8: return launch_qm_m<8, PAIR>(a, s, info);
    default: return TC_NOT_TAKEN;
    }
}

}  // namespace
}  // namespace qgemv
