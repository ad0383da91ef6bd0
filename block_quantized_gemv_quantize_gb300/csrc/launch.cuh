// Internal launch helpers shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qgemv.h"
#include "mmvq.cuh"

namespace qgemv {

struct DeviceInfo {
    int sms;
    int smem_optin;
};

// Per-device properties, queried once per device.
DeviceInfo device_info();

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

template <int FMT, int M, bool TOP1>
int launch_mmvq_m(MmvqArgs a, cudaStream_t s)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    const int NB = a.K / QK;
    const size_t extra = mmvq_smem_bytes<M, TOP1>(0);
    a.KC = mmvq_chunk_blocks(di, M, NB, extra);
    const size_t smem = mmvq_smem_bytes<M, TOP1>(a.KC);
    if (smem > (size_t)di.smem_optin) return QGEMV_UNSUPPORTED_SHAPE;
    auto kern = mmvq_kernel<FMT, M, TOP1>;
    // Opt in to the device's full shared memory once per device.
    static bool opted[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return QGEMV_CUDA_ERROR;
    if (!opted[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin) != cudaSuccess)
            return QGEMV_CUDA_ERROR;
        opted[dev] = true;
    }
    constexpr int R = RowsPerWarp<M>::value;
    const int n_rg = (a.N + R - 1) / R;
    const int n_items = (n_rg + MMVQ_WARPS - 1) / MMVQ_WARPS;
    const int grid = n_items < di.sms ? n_items : di.sms;
    kern<<<grid, MMVQ_THREADS, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

int launch_mmvq_q4_0(const MmvqArgs& a, int M, cudaStream_t s);
int launch_mmvq_q6_k(const MmvqArgs& a, int M, cudaStream_t s);
int launch_lmhead_q6_k(const MmvqArgs& a, int M, cudaStream_t s);

int launch_quantize_q8_1(const float* x, int64_t ldx, void* xq, int M, int K, cudaStream_t s);
int launch_qpack_q4_0(const void* canon, void* pack, int N, int K, cudaStream_t s);
int launch_qpack_q6_k(const void* canon, void* pack, int N, int K, cudaStream_t s);
int launch_argmax_rows(const float* y, int64_t ldy, int32_t* ids, Top1Workspace* ws, int M, int N, cudaStream_t s);
int launch_block_dots(int fmt, const void* w_pack, const void* xq, int32_t* out, int M, int K, int N, cudaStream_t s);

}  // namespace qgemv
