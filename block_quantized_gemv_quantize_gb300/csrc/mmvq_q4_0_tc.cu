// Host side of the tensor-core Q4_0 MMVQ: tensor maps over the packed
// weight, the launch plan (cluster size, ring depth) and the launch, for
// M = 1..17, one weight or a pair.
#include <cudaTypedefs.h>

#include <atomic>

#include "launch.cuh"
#include "mmvq_tc.cuh"

namespace qgemv {

namespace {

std::atomic<int> g_tc_enabled{1};

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Tensor maps of a packed Q4_0 weight whose groups and chunks are all whole
// (N % 16 == 0, K % 1024 == 0): every group-chunk is 2304 B, codes
// nib[4 rows][32 blocks][16 B] then scales d[32 blocks][4 rows].
//   codes:  bytes of a row's chunk (512) x row (4) x chunk (nch) x group,
//           box 128 B x 4 rows x 1 chunk x 4 groups = 16 rows x 8 blocks,
//           128-byte swizzled (a job takes two);
//   scales: bytes of the chunk's scales (256) x chunk x group, box jb * 8 B
//           x 1 x 4 groups = a job's 16 rows x jb blocks.
bool q4_0_tensor_maps(const void* w, int N, int K, int jb, CUtensorMap* nib, CUtensorMap* d)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const Layout L = make_layout(FMT_Q4_0, N, K);
    const cuuint64_t gc = (cuuint64_t)L.chunk_bytes(GROUP, 0);  // 2304
    const cuuint64_t gs = (cuuint64_t)L.nch * gc;
    {
        const cuuint64_t dims[4] = {(cuuint64_t)CHUNK * 16, GROUP, (cuuint64_t)L.nch, (cuuint64_t)L.n_groups};
        const cuuint64_t strides[3] = {(cuuint64_t)CHUNK * 16, gc, gs};
        const cuuint32_t box[4] = {TC_LINE_JB * 16, GROUP, 1, TC_ROWS / GROUP};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(w), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)CHUNK * GROUP * 2, (cuuint64_t)L.nch, (cuuint64_t)L.n_groups};
        const cuuint64_t strides[2] = {gc, gs};
        const cuuint32_t box[3] = {(cuuint32_t)jb * GROUP * 2, 1, TC_ROWS / GROUP};
        const cuuint32_t es[3] = {1, 1, 1};
        void* base = static_cast<uint8_t*>(const_cast<void*>(w)) + (size_t)GROUP * CHUNK * 16;
        if (enc(d, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

struct TcPlan {
    int C, grid, S, jb, nkb_max, out_tiles;
    size_t smem;
};

constexpr int TC_CLUSTERS[4] = {1, 2, 4, 8};

template <int M, bool PAIR>
cudaError_t tc_launch(const TcPlan& p, const TcArgs& a, const CUtensorMap& n0, const CUtensorMap& d0,
                      const CUtensorMap& n1, const CUtensorMap& d1, unsigned int* timeouts, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(TC_THREADS);
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
    return cudaLaunchKernelEx(&cfg, mmvq_q4_0_tc_kernel<M, PAIR>, a, n0, d0, n1, d1, timeouts);
}

// Clusters of C CTAs of this kernel (one per SM) that can be resident at once.
template <int M, bool PAIR>
int tc_max_clusters(int dev, int ci, size_t smem)
{
    static int cache[64][4];
    static bool have[64][4];
    if (!have[dev][ci]) {
        const int C = TC_CLUSTERS[ci];
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C);
        cfg.blockDim = dim3(TC_THREADS);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mmvq_q4_0_tc_kernel<M, PAIR>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cache[dev][ci] = n;
        have[dev][ci] = true;
    }
    return cache[dev][ci];
}

// The cheapest plan over job sizes JB (16 or 8 blocks) and cluster sizes C:
// the largest per-CTA job count over 16 warps (the critical path) in units of
// 8 blocks, where a 16-block job counts 0.85 x 2 units (measured: it halves
// the per-job copy issue and loop overhead), plus two units for the
// cross-CTA combine when C > 1.  Returns false when nothing fits.
template <int M, bool PAIR>
bool tc_plan(const DeviceInfo& di, int dev, int K, int N, int N2, TcPlan& best)
{
    const int W = TC_THREADS / 32;
    const int NB = K / QK;
    const int64_t T = N / TC_ROWS + (PAIR ? N2 / TC_ROWS : 0);
    double best_cost = 0.0;
    bool found = false;
    for (int jb = 2 * TC_LINE_JB; jb >= TC_LINE_JB; jb -= TC_LINE_JB) {
        const int njb = NB / jb;
        for (int ci = 0; ci < 4; ++ci) {
            const int C = TC_CLUSTERS[ci];
            if (njb < C) break;
            const int jpt = (njb + C - 1) / C;
            const int nkb = jpt * jb;
            if (nkb * ((M + 7) / 8) * 8 > tc_stage_items(M) * TC_THREADS) continue;  // staging items per thread
            // shared memory at the deepest ring that fits
            int64_t ncl = C == 1 ? di.sms : 0;
            if (C > 1) {
                if (tc_smem(M, W, 2, nkb, 0, jb).bytes > (uint32_t)di.smem_optin) continue;
                ncl = tc_max_clusters<M, PAIR>(dev, ci, (size_t)di.smem_optin);
                if (ncl <= 0) continue;
            }
            if (ncl > T) ncl = T;
            const int tiles = (int)((T + ncl - 1) / ncl);
            const int out_tiles = C > 1 ? tiles : 0;
            int S = 0;
            for (int s = TC_MAX_STAGES; s >= 2; --s) {
                if (tc_smem(M, W, s, nkb, out_tiles, jb).bytes <= (uint32_t)di.smem_optin) {
                    S = s;
                    break;
                }
            }
            if (S == 0) continue;
            const double unit = jb > TC_LINE_JB ? 0.85 * jb / TC_LINE_JB : 1.0;
            const double cost = (double)(((int64_t)tiles * jpt + W - 1) / W) * unit + (C > 1 ? 2.0 : 0.0);
            if (!found || cost < best_cost - 1e-9) {
                found = true;
                best_cost = cost;
                best.C = C;
                best.grid = (int)(ncl * C);
                best.S = S;
                best.jb = jb;
                best.nkb_max = nkb;
                best.out_tiles = out_tiles;
                best.smem = tc_smem(M, W, S, nkb, out_tiles, jb).bytes;
            }
        }
    }
    return found;
}

// Opt the kernel in to the device's full shared memory (once per device);
// returns the device's timeout counter, or null on failure.
template <int M, bool PAIR>
unsigned int* tc_prepare(const DeviceInfo& di, int dev)
{
    static bool opted[64];
    static unsigned int* timeouts[64];
    if (!opted[dev]) {
        if (cudaFuncSetAttribute(mmvq_q4_0_tc_kernel<M, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 di.smem_optin) != cudaSuccess)
            return nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&timeouts[dev]), g_wait_timeouts) != cudaSuccess)
            return nullptr;
        opted[dev] = true;
    }
    return timeouts[dev];
}

// info (when not null): {1, cluster size, grid, ring stages} of the plan.
template <int M, bool PAIR>
int launch_tc_m(const MmvqArgs& m, cudaStream_t s, int* info)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QGEMV_CUDA_ERROR;
    unsigned int* timeouts = tc_prepare<M, PAIR>(di, dev);
    if (!timeouts) return QGEMV_CUDA_ERROR;
    TcPlan p{};
    if (!tc_plan<M, PAIR>(di, dev, m.K, m.N, PAIR ? m.N2 : 0, p)) return TC_NOT_TAKEN;
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
    if (tc_launch<M, PAIR>(p, a, n0, d0, n1, d1, timeouts, s) != cudaSuccess) return QGEMV_CUDA_ERROR;
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

int set_q4_0_tensor_cores(int enable) { return g_tc_enabled.exchange(enable ? 1 : 0); }

int launch_mmvq_q4_0_tc(const MmvqArgs& a, int M, bool pair, cudaStream_t s, int* info)
{
    if (!g_tc_enabled.load()) return TC_NOT_TAKEN;
    // Below 5 rows the SIMT kernels are as fast or faster (measured on GB300:
    // M <= 4 loses up to 12% on the tensor cores, M >= 5 gains up to 34%).
    if (M < TC_MIN_M) return TC_NOT_TAKEN;
    if (a.N % TC_ROWS || (pair && a.N2 % TC_ROWS) || a.K % (CHUNK * QK)) return TC_NOT_TAKEN;
    return pair ? launch_tc<true>(a, M, s, info) : launch_tc<false>(a, M, s, info);
}

unsigned int take_wait_timeouts_q4_0_tc() { return take_wait_timeouts_tu(); }

}  // namespace qgemv
