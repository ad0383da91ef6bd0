// Internal launch helpers shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/qgemv.h"
#include "mmvq.cuh"

namespace qgemv {

struct DeviceInfo {
    int sms;
    int smem_optin;
};

// Per-device properties, queried once per device.
DeviceInfo device_info();

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream drains; it orders itself after that
// kernel with pdl_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// The library-wide count of warps that gave up waiting for their data (a
// bounded wait ran out): the device address kernels add to (system-scope
// atomics), host memory mapped into the device address space when that could
// be set up, a device word otherwise; null if neither could.
unsigned int* wait_timeout_counter();
// Whether a kernel gave up waiting since the count was last taken (false when
// the counter is a device word, which the host cannot read without a copy).
bool wait_timeouts_pending();
// A test-only request (qgemv_debug_drop_next_copy) taken by the next launch of
// the small-M Q4_0 kernel: 1 once, then 0.
int take_drop_request();
// Debug build only (test hook): whether the next ring-kernel launch should
// move one output store out of its extent, for its bounds check to catch.
int take_plant_request();

// Largest multiple-of-32 block chunk of activation that fits in shared memory
// next to `extra` bytes (all of K when it fits).
inline int mmvq_chunk_blocks(const DeviceInfo& di, int M, int NB, size_t extra)
{
    const size_t budget = (size_t)di.smem_optin - extra - 1024;
    const size_t per_block = (size_t)M * ACT_BYTES_PER_BLOCK;
    size_t kc = budget / per_block;
    if ((size_t)NB <= kc) return NB;
    kc = (kc / 32) * 32;
    return kc < 32 ? 32 : (int)kc;
}

constexpr int MAX_RING_STAGES = 8;

// Launch configuration of one MMVQ call.
struct MmvqPlan {
    bool ring;
    int grid, warps, stages, parts, KC;
    size_t smem;
};

// K parts per row group for the ring kernel (part p: chunks p nch / P ..
// (p + 1) nch / P - 1).  A CTA's G groups become G * P items dealt
// round-robin to its W warps, so it runs ceil(G P / W) rounds of at most
// ceil(nch / P) jobs plus one reduction (about a third of a job) each; take
// the P with the fewest job-times (the smallest on a tie).  The top-1 kernel
// keeps P = 1.
inline int ring_parts(int64_t groups_per_cta, int nch, int max_warps, bool top1)
{
    if (top1) return 1;
    int best_p = 1;
    double best = 0.0;
    for (int P = 1; P <= nch && P <= 32; ++P) {
        const int64_t items = groups_per_cta * P;
        const int64_t w = items < max_warps ? items : max_warps;
        const int64_t rounds = (items + w - 1) / w;
        const double cost = (double)rounds * ((double)((nch + P - 1) / P) + 0.35);
        if (P == 1 || cost < best - 1e-9) {
            best = cost;
            best_p = P;
        }
    }
    return best_p;
}

// N2 > 0: a second weight of N2 rows and the same K, whose row groups the
// ring kernel takes after the first's.
template <int FMT, int M, bool TOP1, bool PAIR = false, bool TOPK = false>
MmvqPlan mmvq_plan(const DeviceInfo& di, int K, int N, int N2 = 0)
{
    const Layout L = make_layout(FMT, N, K);
    const int max_warps = MmvqThreads<FMT, M, TOP1, TOPK>::value / 32;
    MmvqPlan p{};
    const int64_t n_groups = L.n_groups + (N2 > 0 ? ((int64_t)N2 + GROUP - 1) / GROUP : 0);
    p.grid = n_groups < di.sms ? (int)n_groups : di.sms;
    const int64_t per_cta = (n_groups + p.grid - 1) / p.grid;  // groups
    p.parts = ring_parts(per_cta, L.nch, max_warps, TOP1);
    const int64_t items = per_cta * p.parts;
    p.warps = items < max_warps ? (int)items : max_warps;
    const size_t act = RingAct<FMT, M>::bytes(L.NB);
    const size_t extra = ring_extra_bytes<M, TOP1, PAIR, TOPK>((int)per_cta, p.parts, max_warps);
    const size_t stage = (size_t)L.chunk_bytes(GROUP, 0) + 8;  // a group-chunk and its mbarrier
    const size_t fixed = act + extra + 128;
    long long s = fixed < (size_t)di.smem_optin ? (long long)(((size_t)di.smem_optin - fixed) / (p.warps * stage)) : 0;
    if (s < 2 && fixed < (size_t)di.smem_optin) {
        // fewer warps with two stages each, if at least four fit
        const long long w = (long long)(((size_t)di.smem_optin - fixed) / (2 * stage));
        if (w >= 4) {
            p.warps = (int)(w < p.warps ? w : p.warps);
            s = 2;
        }
    }
    if (s > MAX_RING_STAGES) s = MAX_RING_STAGES;
    if (s >= 2) {
        p.ring = true;
        p.stages = (int)s;
        p.KC = L.NB;
        p.smem = (size_t)p.warps * p.stages * stage + act + extra;
        return p;
    }
    p.ring = false;  // (the lock-step kernel takes one weight at a time)
    p.parts = 1;
    p.warps = max_warps;
    const int64_t n_items = (L.n_groups + p.warps - 1) / p.warps;
    p.grid = n_items < di.sms ? (int)n_items : di.sms;
    const size_t ex = TOP1 ? top1_scratch_bytes(p.warps) : 0;
    p.KC = mmvq_chunk_blocks(di, M, L.NB, ex);
    p.stages = 0;
    p.smem = (size_t)M * p.KC * ACT_BYTES_PER_BLOCK + ex;
    return p;
}

// The most CTAs a top-k launch may have: its workspace holds one list per CTA.
constexpr int TOPK_MAX_CTAS = 256;

template <int FMT, int M, bool TOP1, bool PAIR, bool RES = false, bool TOPK = false>
int launch_mmvq_pm(MmvqArgs a, cudaStream_t s)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QGEMV_CUDA_ERROR;
    const MmvqPlan p = mmvq_plan<FMT, M, TOP1, PAIR, TOPK>(di, a.K, a.N, PAIR ? a.N2 : 0);
    if (p.smem > (size_t)di.smem_optin) return QGEMV_UNSUPPORTED_SHAPE;
    // top-k runs on the ring kernel only, with one list per CTA in the workspace
    if (TOPK && (!p.ring || p.grid > TOPK_MAX_CTAS)) return QGEMV_UNSUPPORTED_SHAPE;
    a.KC = p.KC;
    a.stages = p.stages;
    a.parts = p.parts;
#ifdef QGEMV_BOUNDS_CHECK
    a.plant_bad_store = p.ring && !TOP1 ? take_plant_request() : 0;
#endif
    // Opt in to the device's full shared memory once per device and kernel
    // (call_once: concurrent first calls from several host threads are safe).
    static std::once_flag once_ring[64], once_lock[64];
    static bool ok_ring[64], ok_lock[64];
    static unsigned int* timeouts[64];
    if (p.ring) {
        auto kern = mmvq_ring_kernel<FMT, M, TOP1, PAIR, RES, TOPK>;
        std::call_once(once_ring[dev], [&]() {
            timeouts[dev] = wait_timeout_counter();
            ok_ring[dev] =
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin) == cudaSuccess &&
                timeouts[dev] != nullptr;
            if (!ok_ring[dev]) cudaGetLastError();
        });
        if (!ok_ring[dev]) return QGEMV_CUDA_ERROR;
        if (launch_pdl(kern, dim3(p.grid), dim3(p.warps * 32), p.smem, s, a, timeouts[dev]) != cudaSuccess)
            return QGEMV_CUDA_ERROR;
    } else if constexpr (!TOPK) {
        auto kern = mmvq_lockstep_kernel<FMT, M, TOP1, RES>;
        std::call_once(once_lock[dev], [&]() {
            ok_lock[dev] =
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin) == cudaSuccess;
            if (!ok_lock[dev]) cudaGetLastError();
        });
        if (!ok_lock[dev]) return QGEMV_CUDA_ERROR;
        unsigned int* status = wait_timeout_counter();
        if (launch_pdl(kern, dim3(p.grid), dim3(p.warps * 32), p.smem, s, a, status) != cudaSuccess)
            return QGEMV_CUDA_ERROR;
        if (PAIR) {  // the lock-step kernel takes the second weight in a launch of its own
            MmvqArgs b = a;
            b.w_pack = a.w_pack2;
            b.y = a.y2;
            b.N = a.N2;
            b.w_pack2 = nullptr;
            b.y2 = nullptr;
            b.N2 = 0;
            const MmvqPlan p2 = mmvq_plan<FMT, M, TOP1>(di, b.K, b.N);
            b.KC = p2.KC;
            if (launch_pdl(kern, dim3(p2.grid), dim3(p2.warps * 32), p2.smem, s, b, status) != cudaSuccess)
                return QGEMV_CUDA_ERROR;
        }
    }
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

// One weight (a.N2 == 0); the pair form is instantiated only for Q4_0 (the
// gate/up projections), via launch_mmvq_pm<..., true> directly.
template <int FMT, int M, bool TOP1>
int launch_mmvq_m(MmvqArgs a, cudaStream_t s)
{
    return launch_mmvq_pm<FMT, M, TOP1, false>(a, s);
}

int launch_mmvq_q4_0(const MmvqArgs& a, int M, cudaStream_t s);
// The tensor-core Q4_0 path (one weight or a pair); TC_NOT_TAKEN when it is
// switched off or the shape is not one it takes (the caller then uses the
// SIMT kernels).
constexpr int TC_NOT_TAKEN = 1;
// info (when not null): nothing is launched; the plan is written instead.
int launch_mmvq_q4_0_tc(const MmvqArgs& a, int M, bool pair, cudaStream_t s, int* info = nullptr);
int set_q4_0_tensor_cores(int mode);
// The small-M tensor-core Q4_0 path (M <= 8, N % 16 == 0, K % 1024 == 0,
// checked by the caller); TC_NOT_TAKEN when no launch plan fits.
int launch_mmvq_q4_0_mma(const MmvqArgs& a, int M, bool pair, cudaStream_t s, int* info = nullptr);
// The tensor-core Q6_K path (M >= TC_Q6_K_MIN_M, N % 16 == 0, K % 1024 == 0);
// TC_NOT_TAKEN otherwise.
int launch_mmvq_q6_k_tc(const MmvqArgs& a, int M, cudaStream_t s, int* info = nullptr);
int set_q6_k_tensor_cores(int mode);
int launch_mmvq_q4_0_pair(const MmvqArgs& a, int M, cudaStream_t s);
// y = W x + residual on the SIMT kernels; the residual travels in a.x / a.ldx
int launch_mmvq_q4_0_residual(const MmvqArgs& a, int M, cudaStream_t s);
int launch_mmvq_q6_k(const MmvqArgs& a, int M, cudaStream_t s);
// Q8_0 (tensor cores, its own pack); QGEMV_UNSUPPORTED_SHAPE when no plan fits
int launch_mmvq_q8_0(const MmvqArgs& a, int M, cudaStream_t s, int* info = nullptr);
int launch_qpack_q8_0(const void* canon, void* pack, int N, int K, cudaStream_t s);
int launch_mmvq_q4_k(const MmvqArgs& a, int M, cudaStream_t s, int* info = nullptr);
int launch_qpack_q4_k(const void* canon, void* pack, int N, int K, cudaStream_t s);
int launch_mmvq_q5_k(const MmvqArgs& a, int M, cudaStream_t s, int* info = nullptr);
int launch_qpack_q5_k(const void* canon, void* pack, int N, int K, cudaStream_t s);
int launch_lmhead_q6_k(const MmvqArgs& a, int M, cudaStream_t s);
// The top-k form (a.topk in 1..TOPK_MAX, a.topk_lists sized for TOPK_MAX_CTAS
// lists); QGEMV_UNSUPPORTED_SHAPE where the activation does not fit the ring
// kernel's shared memory.
int launch_lmhead_q6_k_topk(const MmvqArgs& a, int M, cudaStream_t s);
// The launch plan of the fused LM-head kernel: {1 ring / 0 lock-step, grid,
// warps, ring stages}.
int lmhead_q6_k_plan(int M, int K, int N, int* info);

int launch_quantize_q8_1(const float* x, int64_t ldx, void* xq, int M, int K, cudaStream_t s);
int launch_rmsnorm_quantize_q8_1(const float* x, int64_t ldx, const float* gamma, float eps, void* xq, int M, int K,
                                 cudaStream_t s);
int launch_qpack_q4_0(const void* canon, void* pack, int N, int K, cudaStream_t s);
int launch_qpack_q6_k(const void* canon, void* pack, int N, int K, cudaStream_t s);
int launch_argmax_rows(const float* y, int64_t ldy, int32_t* ids, Top1Workspace* ws, int M, int N, cudaStream_t s);
int launch_block_dots(int fmt, const void* w_pack, const void* xq, int32_t* out, int M, int K, int N, cudaStream_t s);

}  // namespace qgemv
