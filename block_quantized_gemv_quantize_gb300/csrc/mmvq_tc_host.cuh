// Host side shared by the tensor-core MMVQ launchers: the launch plan
// (job size, cluster size, ring depth), cluster occupancy, the launch and
// the per-device opt-in.  Included by one translation unit per format.
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "launch.cuh"
#include "mmvq_tc.cuh"

namespace qgemv {
namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
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
// tiles: 16-row tiles per box (the general kernel's boxes hold one; the
// small-M kernel's may hold two).
bool q4_0_tensor_maps(const void* w, int N, int K, int jb, CUtensorMap* nib, CUtensorMap* d, int tiles = 1)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const Layout L = make_layout(FMT_Q4_0, N, K);
    const cuuint64_t gc = (cuuint64_t)L.chunk_bytes(GROUP, 0);  // 2304
    const cuuint64_t gs = (cuuint64_t)L.nch * gc;
    {
        const cuuint64_t dims[4] = {(cuuint64_t)CHUNK * 16, GROUP, (cuuint64_t)L.nch, (cuuint64_t)L.n_groups};
        const cuuint64_t strides[3] = {(cuuint64_t)CHUNK * 16, gc, gs};
        const cuuint32_t box[4] = {TC_LINE_JB * 16, GROUP, 1, (cuuint32_t)(tiles * TC_ROWS / GROUP)};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(nib, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(w), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)CHUNK * GROUP * 2, (cuuint64_t)L.nch, (cuuint64_t)L.n_groups};
        const cuuint64_t strides[2] = {gc, gs};
        const cuuint32_t box[3] = {(cuuint32_t)jb * GROUP * 2, 1, (cuuint32_t)(tiles * TC_ROWS / GROUP)};
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

template <int FMT, int M, bool PAIR>
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
    return cudaLaunchKernelEx(&cfg, mmvq_tc_kernel<FMT, M, PAIR>, a, n0, d0, n1, d1, timeouts);
}

// Clusters of C CTAs of this kernel (one per SM) that can be resident at once.
template <int FMT, int M, bool PAIR>
int tc_max_clusters(int dev, int ci, size_t smem)
{
    static int cache[64][4];
    static std::once_flag once[64][4];
    std::call_once(once[dev][ci], [&]() {
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
        if (cudaOccupancyMaxActiveClusters(&n, mmvq_tc_kernel<FMT, M, PAIR>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cache[dev][ci] = n;
    });
    return cache[dev][ci];
}

// The cheapest plan over job sizes JB (Q4_0: 16 or 8 blocks; Q4_K, Q5_K: the
// same up to M = 8, then 8; Q8_0: 8 or 4; Q6_K: 8)
// and cluster sizes C:
// the largest per-CTA job count over 16 warps (the critical path) in units of
// 8 blocks, where a 16-block Q4_0 job counts 0.85 x 2 units (measured: it
// halves the per-job copy issue and loop overhead) and a 4-block Q8_0 job 0.75
// (its copy issue and loop overhead stay whole), plus two units for the
// cross-CTA combine when C > 1, times the waves when more clusters are
// launched than are resident.  Returns false when nothing fits.
template <int FMT, int M, bool PAIR>
bool tc_plan(const DeviceInfo& di, int dev, int K, int N, int N2, TcPlan& best)
{
    const int W = TC_THREADS / 32;
    const int NB = K / QK;
    const int64_t T = (N + TC_ROWS - 1) / TC_ROWS + (PAIR ? (N2 + TC_ROWS - 1) / TC_ROWS : 0);
    double best_cost = 0.0;
    bool found = false;
    // Q4_0: 16- then 8-block jobs; Q8_0: whole 8-block regions, then halves
    // (Q4_K / Q5_K: 16-block jobs only up to M = 8, where they measured faster
    // at every N; above it they traded ring depth for waves and measured
    // slower about as often as faster)
    const int jb_first = FMT == TCF_Q8_0                                       ? TC_Q8_0_JOB_BLOCKS
                         : FMT == TCF_Q6_K                                     ? TC_LINE_JB
                         : (FMT == TCF_Q4_K || FMT == TCF_Q5_K) && M > 8 ? TC_LINE_JB
                                                                               : 2 * TC_LINE_JB;
    const int jb_last = FMT == TCF_Q8_0 ? TC_Q8_0_JOB_BLOCKS / 2 : TC_LINE_JB;
    const int metab = tc_meta_bytes(FMT);
    for (int jb = jb_first; jb >= jb_last; jb /= 2) {
        if (NB % jb) continue;  // whole jobs only
        const int njb = NB / jb;
        const int nibs = FMT == TCF_Q8_0   ? tc_q8_0_job_bytes(jb)
                         : FMT == TCF_Q6_K ? TC_Q6_K_NIB
                         : FMT == TCF_Q4_K ? TC_Q4_K_JOB * (jb / 8)
                         : FMT == TCF_Q5_K ? TC_Q5_K_JOB * (jb / 8)
                                           : tc_nib_bytes(jb);
        const int dsb = FMT == TCF_Q6_K ? TC_Q6_K_DS : FMT == TCF_Q4_0 ? tc_ds_bytes(jb) : 0;
        for (int ci = 0; ci < 4; ++ci) {
            const int C = TC_CLUSTERS[ci];
            if (njb < C) break;
            const int jpt = (njb + C - 1) / C;
            const int nkb = jpt * jb;
            if (nkb * ((M + 7) / 8) * 8 > tc_stage_items(M) * TC_THREADS) continue;  // staging items per thread
            // shared memory at the deepest ring that fits
            int64_t ncl = C == 1 ? di.sms : 0;
            if (C > 1) {
                if (tc_smem(M, W, 2, nkb, 0, nibs, dsb, metab).bytes > (uint32_t)di.smem_optin) continue;
                ncl = tc_max_clusters<FMT, M, PAIR>(dev, ci, (size_t)di.smem_optin);
                if (ncl <= 0) continue;
            }
            if (ncl > T) ncl = T;
            int64_t ngrid = ncl;  // clusters launched
            int tiles = (int)((T + ncl - 1) / ncl);
            int64_t waves = 1;
            auto deepest = [&](int out_tiles) {
                for (int s = TC_MAX_STAGES; s >= 2; --s)
                    if (tc_smem(M, W, s, nkb, out_tiles, nibs, dsb, metab).bytes <= (uint32_t)di.smem_optin) return s;
                return 0;
            };
            int S = deepest(C > 1 ? tiles : 0);
            if (S == 0 && C > 1) {
                // The combine area of one resident wave's tiles does not fit
                // (very large N): launch more clusters than are resident, in
                // waves, each with as many tiles as the area holds.
                const int64_t per_tile = tc_smem(M, W, 2, nkb, 1, nibs, dsb, metab).bytes - tc_smem(M, W, 2, nkb, 0, nibs, dsb, metab).bytes;
                const int64_t room = (int64_t)di.smem_optin - tc_smem(M, W, 2, nkb, 0, nibs, dsb, metab).bytes;
                const int64_t fit = room / per_tile;
                if (fit >= 1) {
                    ngrid = (T + fit - 1) / fit;
                    tiles = (int)((T + ngrid - 1) / ngrid);
                    waves = (ngrid + ncl - 1) / ncl;
                    S = deepest(tiles);
                }
            }
            if (S == 0) continue;
            const int out_tiles = C > 1 ? tiles : 0;
            const double unit = FMT == TCF_Q8_0 ? (jb < TC_Q8_0_JOB_BLOCKS ? 0.75 : 1.0)
                                : (jb > TC_LINE_JB ? 0.85 * jb / TC_LINE_JB : 1.0);
            const double cost =
                (double)waves * ((double)(((int64_t)tiles * jpt + W - 1) / W) * unit + (C > 1 ? 2.0 : 0.0));
            if (!found || cost < best_cost - 1e-9) {
                found = true;
                best_cost = cost;
                best.C = C;
                best.grid = (int)(ngrid * C);
                best.S = S;
                best.jb = jb;
                best.nkb_max = nkb;
                best.out_tiles = out_tiles;
                best.smem = tc_smem(M, W, S, nkb, out_tiles, nibs, dsb, metab).bytes;
            }
        }
    }
    return found;
}

// Opt the kernel in to the device's full shared memory (once per device);
// returns the device's timeout counter, or null on failure.
template <int FMT, int M, bool PAIR>
unsigned int* tc_prepare(const DeviceInfo& di, int dev)
{
    static std::once_flag once[64];
    static unsigned int* timeouts[64];
    std::call_once(once[dev], [&]() {
        timeouts[dev] = wait_timeout_counter();
        if (cudaFuncSetAttribute(mmvq_tc_kernel<FMT, M, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 di.smem_optin) != cudaSuccess) {
            timeouts[dev] = nullptr;
            cudaGetLastError();
        }
    });
    return timeouts[dev];
}

}  // namespace
}  // namespace qgemv
