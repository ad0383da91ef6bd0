// Host side of the tensor-core Q6_K MMVQ: four tensor maps over the existing
// Q6_K pack (no second weight format), the launch plan and the launch, for
// the activation row counts where the tensor cores beat the dp4a kernel.
#include <atomic>

#include "mmvq_tc_host.cuh"

namespace qgemv {

namespace {

std::atomic<int> g_q6_k_tc_enabled{1};

// Tensor maps of a packed Q6_K weight whose groups and chunks are all whole
// (N % 16 == 0, K % 1024 == 0): every group-chunk is 3360 B = four 832-byte
// row tiles (the code bytes P[32][16 B] and Q[32][8 B], sc[32][2 B]) then
// d[4 rows][4 superblocks] fp16.  The first three maps view the row tiles as bytes (832) x
// row (4) x chunk x group and differ in box and swizzle:
//   P:  box 128 B x 4 x 1 x 4 groups (16 rows x 8 blocks), 128-byte swizzle;
//   Q:  box  64 B x 4 x 1 x 4, 64-byte swizzle;
//   sc: box  16 B x 4 x 1 x 4;
// the fourth views the scale tails as bytes (32) x chunk x group, box 32 B x
// 1 x 4 groups.
bool q6_k_tensor_maps(const void* w, int N, int K, CUtensorMap* ql, CUtensorMap* qh, CUtensorMap* sc,
                      CUtensorMap* d)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const Layout L = make_layout(FMT_Q6_K, N, K);
    const cuuint64_t tile = (cuuint64_t)L.tile(0);             // 832
    const cuuint64_t gc = (cuuint64_t)L.chunk_bytes(GROUP, 0);  // 3360
    const cuuint64_t gs = (cuuint64_t)L.nch * gc;
    const cuuint64_t dims[4] = {tile, GROUP, (cuuint64_t)L.nch, (cuuint64_t)L.n_groups};
    const cuuint64_t strides[3] = {tile, gc, gs};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    struct Box {
        CUtensorMap* map;
        cuuint32_t x;
        CUtensorMapSwizzle sw;
    } boxes[3] = {{ql, 128, CU_TENSOR_MAP_SWIZZLE_128B}, {qh, 64, CU_TENSOR_MAP_SWIZZLE_64B},
                  {sc, 16, CU_TENSOR_MAP_SWIZZLE_NONE}};
    for (const Box& b : boxes) {
        const cuuint32_t box[4] = {b.x, GROUP, 1, TC_ROWS / GROUP};
        if (enc(b.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(w), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, b.sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        const cuuint64_t ddims[3] = {(cuuint64_t)GROUP * 8, (cuuint64_t)L.nch, (cuuint64_t)L.n_groups};
        const cuuint64_t dstrides[2] = {gc, gs};
        const cuuint32_t box[3] = {GROUP * 8, 1, TC_ROWS / GROUP};
        void* base = static_cast<uint8_t*>(const_cast<void*>(w)) + (size_t)GROUP * tile;
        if (enc(d, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, ddims, dstrides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

// info (when not null): {1, cluster size, grid, ring stages} of the plan.
template <int M>
int launch_q6_k_tc_m(const MmvqArgs& m, cudaStream_t s, int* info)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QGEMV_CUDA_ERROR;
    unsigned int* timeouts = tc_prepare<TCF_Q6_K, M, false>(di, dev);
    if (!timeouts) return QGEMV_CUDA_ERROR;
    TcPlan p{};
    if (!tc_plan<TCF_Q6_K, M, false>(di, dev, m.K, m.N, 0, p)) return TC_NOT_TAKEN;
    if (info) {
        info[0] = 1;
        info[1] = p.C;
        info[2] = p.grid;
        info[3] = p.S;
        return QGEMV_OK;
    }
    CUtensorMap ql, qh, sc, d;
    if (!q6_k_tensor_maps(m.w_pack, m.N, m.K, &ql, &qh, &sc, &d)) return QGEMV_CUDA_ERROR;
    TcArgs a{};
    a.xq = m.xq;
    a.y = m.y;
    a.ldy = m.ldy;
    a.K = m.K;
    a.N = m.N;
    a.stages = p.S;
    a.jb = p.jb;
    a.nkb_max = p.nkb_max;
    a.out_tiles = p.out_tiles;
    // the kernel's four map slots: ql, qh (codes), sc, d (scales)
    if (tc_launch<TCF_Q6_K, M, false>(p, a, ql, qh, sc, d, timeouts, s) != cudaSuccess) return QGEMV_CUDA_ERROR;
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

}  // namespace

int set_q6_k_tensor_cores(int mode) { return g_q6_k_tc_enabled.exchange(mode < 0 ? 0 : mode > 2 ? 2 : mode); }

// Where the tensor cores beat the dp4a kernel (GB300, lone calls after an L2
// flush): only when the dp4a kernel has to split K (fewer than 16 row groups
// per SM, N < 9728) and either M >= 12 or K >= 16384 (K = 17408, N = 5120:
// 40 vs 56 us at M = 7, 52 vs 91 us at M = 12; K = 5120, N = 5120: 25 vs
// 27-31 us at M = 12-17, but 21-25 vs 19-23 us at M = 7-9).  At large N the
// f16 activation tile leaves room for only two ring stages per warp and the
// kernel waits on its copies (N = 248320, M = 7: 283 vs 232 us).
static bool q6_k_tc_pays(int M, int K, int N, int sms)
{
    return (int64_t)N < (int64_t)sms * 16 * GROUP && (M >= 12 || K >= 16384);
}

int launch_mmvq_q6_k_tc(const MmvqArgs& a, int M, cudaStream_t s, int* info)
{
    const int mode = g_q6_k_tc_enabled.load();
    if (mode == 0) return TC_NOT_TAKEN;
    if (M < TC_Q6_K_MIN_M) return TC_NOT_TAKEN;
    if (a.N % TC_ROWS || a.K % (CHUNK * QK)) return TC_NOT_TAKEN;
    if (mode == 1 && !q6_k_tc_pays(M, a.K, a.N, device_info().sms)) return TC_NOT_TAKEN;
    switch (M) {
    case 1: return launch_q6_k_tc_m<1>(a, s, info);
    case 2: return launch_q6_k_tc_m<2>(a, s, info);
    case 3: return launch_q6_k_tc_m<3>(a, s, info);
    case 4: return launch_q6_k_tc_m<4>(a, s, info);
    case 5: return launch_q6_k_tc_m<5>(a, s, info);
    case 6: return launch_q6_k_tc_m<6>(a, s, info);
    case 7: return launch_q6_k_tc_m<7>(a, s, info);
    case 8: return launch_q6_k_tc_m<8>(a, s, info);
    case 9: return launch_q6_k_tc_m<9>(a, s, info);
    case 10: return launch_q6_k_tc_m<10>(a, s, info);
    case 11: return launch_q6_k_tc_m<11>(a, s, info);
    case 12: return launch_q6_k_tc_m<12>(a, s, info);
    case 13: return launch_q6_k_tc_m<13>(a, s, info);
    case 14: return launch_q6_k_tc_m<14>(a, s, info);
    case 15: return launch_q6_k_tc_m<15>(a, s, info);
    case 16: return launch_q6_k_tc_m<16>(a, s, info);
    case 17: return launch_q6_k_tc_m<17>(a, s, info);
    default: return TC_NOT_TAKEN;
    }
}


}  // namespace qgemv
