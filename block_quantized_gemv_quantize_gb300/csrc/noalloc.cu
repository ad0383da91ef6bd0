// lmhead_q6_k_top1_noalloc: the fused Q6_K LM-head top-1 for callers that
// cannot hand the library a device workspace.
//
// lmhead_q6_k_top1 needs a small zero-filled workspace (one 64-bit key per
// row plus a completion counter) for its cross-CTA reduction.  Some callers
// cannot allocate device memory at the point where they run this: code that
// executes while another component owns every byte of the device through its
// own pool and forbids side allocations, code on a latency path where a
// cudaMalloc could stall or synchronize the device, or code that is only
// given input and output pointers by its host.  This entry point keeps that
// scratch in a fixed array in this library's device memory instead.
//
// The scratch is a file-scope __device__ array (256 bytes, enough for the
// keys of QGEMV_NOALLOC_MAX_M = 17 rows and the counter); every GPU that
// loads the library holds it until the process exits.  Host code cannot use
// the array's name as a device address, so its device address is looked up
// once per device with cudaGetSymbolAddress, with that device current, on the
// first call made on the device.  The cached address does not survive a
// reset of the device's primary context (cudaDeviceReset reloads the
// library's module); the header tells callers not to use this entry point on
// a device after resetting it.
#include "../../include/qgemv.h"
#include "launch.cuh"

#include <mutex>

namespace qgemv {
namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 256;
static_assert(sizeof(Top1Workspace) <= NOALLOC_SCRATCH_BYTES, "top-1 scratch does not fit");

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[MAX_DEVICES];

// Device address of the scratch array on the current device (looked up once).
int scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return QGEMV_CUDA_ERROR;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QGEMV_CUDA_ERROR;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return QGEMV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace qgemv

using namespace qgemv;

extern "C" int lmhead_q6_k_top1_noalloc(const void* w_pack, const float* x, int64_t ldx, int32_t* ids, int M, int K,
                                        int N, void* stream)
{
    if (wait_timeouts_pending()) return QGEMV_WAIT_TIMEOUT;
    if (!w_pack || !x || !ids) return QGEMV_INVALID_ARG;
    if (M < 1 || K < QK_K || N < 1 || ldx < K) return QGEMV_INVALID_ARG;
    if (M > QGEMV_NOALLOC_MAX_M) return QGEMV_UNSUPPORTED_SHAPE;  // beyond the fixed scratch
    if (K % QK_K) return QGEMV_UNSUPPORTED_SHAPE;
    if (!aligned16(w_pack) || !aligned16(x) || !aligned16(ids)) return QGEMV_MISALIGNED;
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != QGEMV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: clear the keys and the
    // counter that the reduction expects to start at zero.
    if (cudaMemsetAsync(scratch, 0, sizeof(Top1Workspace), s) != cudaSuccess) return QGEMV_CUDA_ERROR;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.x = x;
    a.ldx = ldx;
    a.K = K;
    a.N = N;
    a.ws = static_cast<Top1Workspace*>(scratch);
    a.ids = ids;
    return launch_lmhead_q6_k(a, M, s);
}
