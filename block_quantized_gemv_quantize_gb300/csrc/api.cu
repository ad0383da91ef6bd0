// C ABI entry points: host-side validation, then one enqueue on the caller's
// stream.  Nothing here allocates or synchronizes.  Fail closed: every
// precondition is checked before any work is enqueued ("Q6_K M=6 fused DFlash
// top-1 production record", Exactness and safety contracts: non-matching
// inputs never reach the fused kernel).
#include "../../include/qgemv.h"
#include "launch.cuh"

#include <atomic>
#include <cstdlib>
#include <mutex>

using namespace qgemv;

namespace {

// The wait-timeout counter.  A word of this library's own host memory,
// registered (page-locked and mapped into the device address space) the first
// time a kernel needs it: kernels add to it with system-scope atomics, the
// host reads it without a copy, and every entry point can see, before it
// enqueues anything, that an earlier call's kernel gave up waiting for its
// data.  Where it cannot be registered, a device word stands in, which only
// qgemv_take_wait_timeouts reads (with a copy).
alignas(4096) unsigned int g_status_page[1024];
__device__ unsigned int g_dev_counter[4];
std::once_flag g_counter_once;
unsigned int* g_counter_dev = nullptr;
bool g_counter_mapped = false;
std::atomic<int> g_drop_request{0};
std::atomic<int> g_plant_request{0};
std::atomic<int> g_fail_fused{0};  // test only: fused LM-head calls to refuse

// Takes one refusal request, if any is left.  The environment variable
// QGEMV_FAIL_FUSED=n (test only) adds n requests when the library first
// looks, so that a process can be started with failing fused calls.
std::once_flag g_fail_env_once;

bool take_fused_failure()
{
    std::call_once(g_fail_env_once, []() {
        const char* e = std::getenv("QGEMV_FAIL_FUSED");
        const int n = e ? std::atoi(e) : 0;
        if (n > 0) g_fail_fused.fetch_add(n);
    });
    int v = g_fail_fused.load();
    while (v > 0)
        if (g_fail_fused.compare_exchange_weak(v, v - 1)) return true;
    return false;
}

void counter_setup()
{
    void* p = nullptr;
    if (cudaHostRegister(g_status_page, sizeof(g_status_page), cudaHostRegisterMapped | cudaHostRegisterPortable) ==
            cudaSuccess &&
        cudaHostGetDevicePointer(&p, g_status_page, 0) == cudaSuccess) {
        g_counter_dev = static_cast<unsigned int*>(p);
        g_counter_mapped = true;
        return;
    }
    cudaGetLastError();
    if (cudaGetSymbolAddress(&p, g_dev_counter) == cudaSuccess) g_counter_dev = static_cast<unsigned int*>(p);
    else cudaGetLastError();
}

// An earlier call's kernel gave up waiting and the count was not taken yet.
bool timeouts_pending()
{
    return g_counter_mapped && __atomic_load_n(&g_status_page[0], __ATOMIC_ACQUIRE) != 0;
}

#define QGEMV_FAIL_IF_TIMED_OUT() \
    do {                          \
        if (timeouts_pending()) return QGEMV_WAIT_TIMEOUT; \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int check_mk(int M, int K, int kmult)
{
    if (M < 1 || K < kmult) return QGEMV_INVALID_ARG;
    if (M > QGEMV_MAX_M) return QGEMV_UNSUPPORTED_SHAPE;
    if (K % kmult != 0) return QGEMV_UNSUPPORTED_SHAPE;
    return QGEMV_OK;
}

int check_gemv(const void* w, const void* xq, const void* y, int64_t ldy, int M, int K, int N, int kmult)
{
    if (!w || !xq || !y) return QGEMV_INVALID_ARG;
    int st = check_mk(M, K, kmult);
    if (st) return st;
    if (N < 1 || ldy < N) return QGEMV_INVALID_ARG;
    if (!aligned16(w) || !aligned16(xq) || !aligned16(y)) return QGEMV_MISALIGNED;
    return QGEMV_OK;
}

size_t top1_ws_bytes() { return sizeof(Top1Workspace); }

// Whether the fp32 matrices [M][lda] at a and [M][ldb] at b share any byte
// (other than being the same matrix).
bool ranges_overlap(const float* a, int64_t lda, const float* b, int64_t ldb, int M, int N)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    const uintptr_t a1 = a0 + (uintptr_t)(((int64_t)(M - 1) * lda + N) * 4);
    const uintptr_t b1 = b0 + (uintptr_t)(((int64_t)(M - 1) * ldb + N) * 4);
    return a0 < b1 && b0 < a1;
}

// lmhead workspace: the top-1 keys and counter, then (from byte
// LMHEAD_Q8_OFFSET) the Q8_1 copy of x that the pre-pass writes.
constexpr size_t LMHEAD_Q8_OFFSET = 256;
static_assert(sizeof(Top1Workspace) <= LMHEAD_Q8_OFFSET, "top-1 scratch does not fit");
size_t lmhead_ws_bytes(int M, int K)
{
    return LMHEAD_Q8_OFFSET + (((size_t)(M > 0 ? M : 0) * (size_t)(K > 0 ? K / QK : 0) * Q8_1_BYTES + 15) & ~(size_t)15);
}

// Top-k workspace: the lmhead workspace, then (256-byte aligned) one list of
// k keys per row for each CTA, at most TOPK_MAX_CTAS CTAs and never more than
// the row groups of N.
static_assert(QGEMV_TOPK_MAX == TOPK_MAX, "top-k bound");
size_t topk_lists_offset(int M, int K) { return (lmhead_ws_bytes(M, K) + 255) & ~(size_t)255; }
size_t topk_ws_bytes(int M, int K, int N, int k)
{
    const int64_t groups = N > 0 ? ((int64_t)N + GROUP - 1) / GROUP : 0;
    const int64_t ctas = groups < TOPK_MAX_CTAS ? groups : TOPK_MAX_CTAS;
    return topk_lists_offset(M, K) + (size_t)ctas * (size_t)(M > 0 ? M : 0) * (size_t)(k > 0 ? k : 0) * 8;
}

}  // namespace

extern "C" {

const char* qgemv_status_string(int status)
{
    switch (status) {
    case QGEMV_OK: return "ok";
    case QGEMV_INVALID_ARG: return "invalid argument (null pointer, or M/K/N/leading dimension out of range)";
    case QGEMV_UNSUPPORTED_SHAPE: return "unsupported shape (M > 17, or K not a multiple of the block size)";
    case QGEMV_MISALIGNED: return "a device pointer is not 16-byte aligned";
    case QGEMV_WORKSPACE_TOO_SMALL: return "workspace too small";
    case QGEMV_CUDA_ERROR: return "CUDA error (launch or device query failed)";
    case QGEMV_WAIT_TIMEOUT:
        return "a kernel of an earlier call gave up waiting for its data, so that call's outputs are not valid "
               "(qgemv_take_wait_timeouts reads and clears the count)";
    default: return "unknown status";
    }
}

size_t q8_1_bytes(int M, int K) { return (M < 0 || K < 0) ? 0 : (size_t)M * (size_t)(K / QK) * Q8_1_BYTES; }
size_t q4_0_pack_bytes(int N, int K)
{
    return (N < 1 || K < QK) ? 0 : (size_t)make_layout(FMT_Q4_0, N, K).total_bytes();
}
size_t q8_0_pack_bytes(int N, int K)
{
    if (N < 1 || K < 256 || K % 256) return 0;
    return (size_t)((N + 15) / 16) * (size_t)(K / 256) * 4352;
}

size_t q4_k_pack_bytes(int N, int K)
{
    if (N < 1 || K < QK_K || K % QK_K) return 0;
    return (size_t)((N + 15) / 16) * (size_t)(K / QK_K) * 2368;
}

size_t q5_k_pack_bytes(int N, int K)
{
    if (N < 1 || K < QK_K || K % QK_K) return 0;
    return (size_t)((N + 15) / 16) * (size_t)(K / QK_K) * 2880;
}

size_t q6_k_pack_bytes(int N, int K)
{
    return (N < 1 || K < QK_K) ? 0 : (size_t)make_layout(FMT_Q6_K, N, K).total_bytes();
}
size_t lmhead_q6_k_top1_workspace_bytes(int M, int K, int) { return lmhead_ws_bytes(M, K); }
size_t argmax_f32_rows_workspace_bytes(int, int) { return top1_ws_bytes(); }
size_t lmhead_q6_k_topk_workspace_bytes(int M, int K, int N, int k) { return topk_ws_bytes(M, K, N, k); }

int quantize_q8_1(const float* x, int64_t ldx, void* xq, int M, int K, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!x || !xq) return QGEMV_INVALID_ARG;
    int st = check_mk(M, K, QK);
    if (st) return st;
    if (ldx < K) return QGEMV_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq)) return QGEMV_MISALIGNED;
    return launch_quantize_q8_1(x, ldx, xq, M, K, as_stream(stream));
}

int rmsnorm_quantize_q8_1(const float* x, int64_t ldx, const float* gamma, float eps, void* xq, int M, int K,
                          void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!x || !gamma || !xq) return QGEMV_INVALID_ARG;
    int st = check_mk(M, K, QK);
    if (st) return st;
    if (ldx < K || !(eps >= 0.0f) || eps > 3.0e38f) return QGEMV_INVALID_ARG;
    if (K >= (1 << 24)) return QGEMV_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(xq)) return QGEMV_MISALIGNED;
    return launch_rmsnorm_quantize_q8_1(x, ldx, gamma, eps, xq, M, K, as_stream(stream));
}

int qpack_q8_0(const void* w_canon, void* w_pack, int N, int K, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!w_canon || !w_pack || N < 1 || K < 256) return QGEMV_INVALID_ARG;
    if (K % 256) return QGEMV_UNSUPPORTED_SHAPE;
    if (!aligned16(w_pack) || (reinterpret_cast<uintptr_t>(w_canon) & 1u)) return QGEMV_MISALIGNED;
    return launch_qpack_q8_0(w_canon, w_pack, N, K, as_stream(stream));
}

int qgemv_q8_0(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    int st = check_gemv(w_pack, xq, y, ldy, M, K, N, 256);
    if (st) return st;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.ldy = ldy;
    a.K = K;
    a.N = N;
    return launch_mmvq_q8_0(a, M, as_stream(stream));
}

int qpack_q4_k(const void* w_canon, void* w_pack, int N, int K, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!w_canon || !w_pack || N < 1 || K < QK_K) return QGEMV_INVALID_ARG;
    if (K % QK_K) return QGEMV_UNSUPPORTED_SHAPE;
    if (!aligned16(w_pack)) return QGEMV_MISALIGNED;
    return launch_qpack_q4_k(w_canon, w_pack, N, K, as_stream(stream));
}

int qgemv_q4_k(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    int st = check_gemv(w_pack, xq, y, ldy, M, K, N, QK_K);
    if (st) return st;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.ldy = ldy;
    a.K = K;
    a.N = N;
    return launch_mmvq_q4_k(a, M, as_stream(stream));
}

int qpack_q5_k(const void* w_canon, void* w_pack, int N, int K, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!w_canon || !w_pack || N < 1 || K < QK_K) return QGEMV_INVALID_ARG;
    if (K % QK_K) return QGEMV_UNSUPPORTED_SHAPE;
    if (!aligned16(w_pack)) return QGEMV_MISALIGNED;
    return launch_qpack_q5_k(w_canon, w_pack, N, K, as_stream(stream));
}

int qgemv_q5_k(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    int st = check_gemv(w_pack, xq, y, ldy, M, K, N, QK_K);
    if (st) return st;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.ldy = ldy;
    a.K = K;
    a.N = N;
    return launch_mmvq_q5_k(a, M, as_stream(stream));
}

int qpack_q4_0(const void* w_canon, void* w_pack, int N, int K, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!w_canon || !w_pack || N < 1 || K < QK) return QGEMV_INVALID_ARG;
    if (K % QK) return QGEMV_UNSUPPORTED_SHAPE;
    if (!aligned16(w_canon) || !aligned16(w_pack)) return QGEMV_MISALIGNED;
    return launch_qpack_q4_0(w_canon, w_pack, N, K, as_stream(stream));
}

int qpack_q6_k(const void* w_canon, void* w_pack, int N, int K, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!w_canon || !w_pack || N < 1 || K < QK_K) return QGEMV_INVALID_ARG;
    if (K % QK_K) return QGEMV_UNSUPPORTED_SHAPE;
    if (!aligned16(w_canon) || !aligned16(w_pack)) return QGEMV_MISALIGNED;
    return launch_qpack_q6_k(w_canon, w_pack, N, K, as_stream(stream));
}

int qgemv_q4_0(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    int st = check_gemv(w_pack, xq, y, ldy, M, K, N, QK);
    if (st) return st;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.ldy = ldy;
    a.K = K;
    a.N = N;
    const int tc = launch_mmvq_q4_0_tc(a, M, false, as_stream(stream));
    if (tc != TC_NOT_TAKEN) return tc;
    return launch_mmvq_q4_0(a, M, as_stream(stream));
}

int qgemv_q4_0_residual(const void* w_pack, const void* xq, const float* residual, int64_t ldr, float* y, int64_t ldy,
                        int M, int K, int N, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    int st = check_gemv(w_pack, xq, y, ldy, M, K, N, QK);
    if (st) return st;
    if (!residual || ldr < N) return QGEMV_INVALID_ARG;
    if (!aligned16(residual)) return QGEMV_MISALIGNED;
    if (residual == y ? ldr != ldy : ranges_overlap(residual, ldr, y, ldy, M, N)) return QGEMV_INVALID_ARG;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.ldy = ldy;
    a.K = K;
    a.N = N;
    a.x = residual;  // the residual instantiations read it from the activation field
    a.ldx = ldr;
    const int tc = launch_mmvq_q4_0_tc(a, M, false, as_stream(stream));
    if (tc != TC_NOT_TAKEN) return tc;
    return launch_mmvq_q4_0_residual(a, M, as_stream(stream));
}

int qgemv_q4_0_pair(const void* w_pack_a, const void* w_pack_b, const void* xq, float* y_a, float* y_b, int64_t ldy,
                    int M, int K, int N_a, int N_b, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    int st = check_gemv(w_pack_a, xq, y_a, ldy, M, K, N_a, QK);
    if (st) return st;
    st = check_gemv(w_pack_b, xq, y_b, ldy, M, K, N_b, QK);
    if (st) return st;
    MmvqArgs a{};
    a.w_pack = w_pack_a;
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y_a;
    a.ldy = ldy;
    a.K = K;
    a.N = N_a;
    a.w_pack2 = w_pack_b;
    a.y2 = y_b;
    a.N2 = N_b;
    const int tc = launch_mmvq_q4_0_tc(a, M, true, as_stream(stream));
    if (tc != TC_NOT_TAKEN) return tc;
    return launch_mmvq_q4_0_pair(a, M, as_stream(stream));
}

int qgemv_q6_k(const void* w_pack, const void* xq, float* y, int64_t ldy, int M, int K, int N, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    int st = check_gemv(w_pack, xq, y, ldy, M, K, N, QK_K);
    if (st) return st;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.xq = static_cast<const uint8_t*>(xq);
    a.y = y;
    a.ldy = ldy;
    a.K = K;
    a.N = N;
    st = launch_mmvq_q6_k_tc(a, M, as_stream(stream));
    if (st != TC_NOT_TAKEN) return st;
    return launch_mmvq_q6_k(a, M, as_stream(stream));
}

int lmhead_q6_k_top1(const void* w_pack, const float* x, int64_t ldx, int32_t* ids, void* workspace,
                     size_t ws_bytes, int M, int K, int N, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!w_pack || !x || !ids || !workspace) return QGEMV_INVALID_ARG;
    int st = check_mk(M, K, QK_K);
    if (st) return st;
    if (N < 1 || ldx < K) return QGEMV_INVALID_ARG;
    if (ws_bytes < lmhead_ws_bytes(M, K)) return QGEMV_WORKSPACE_TOO_SMALL;
    if (!aligned16(w_pack) || !aligned16(x) || !aligned16(ids) || !aligned16(workspace)) return QGEMV_MISALIGNED;
    if (take_fused_failure()) return QGEMV_CUDA_ERROR;  // test only: nothing enqueued
    // Pre-pass: x -> Q8_1 in the workspace (the same kernel as quantize_q8_1),
    // then the MMVQ kernel with the top-1 epilogue reads that copy.
    uint8_t* xq = static_cast<uint8_t*>(workspace) + LMHEAD_Q8_OFFSET;
    cudaStream_t s = as_stream(stream);
    st = launch_quantize_q8_1(x, ldx, xq, M, K, s);
    if (st != QGEMV_OK) return st;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.x = x;
    a.ldx = ldx;
    a.xq = xq;
    a.K = K;
    a.N = N;
    a.ws = static_cast<Top1Workspace*>(workspace);
    a.ids = ids;
    return launch_lmhead_q6_k(a, M, s);
}

int lmhead_q6_k_candmax(const void* w_pack, const float* x, int64_t ldx, const int32_t* cand, int32_t* ids,
                        float* top_vals, float* cand_vals, void* workspace, size_t ws_bytes, int M, int K, int N,
                        void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!w_pack || !x || !cand || !ids || !top_vals || !cand_vals || !workspace) return QGEMV_INVALID_ARG;
    int st = check_mk(M, K, QK_K);
    if (st) return st;
    if (N < 1 || ldx < K) return QGEMV_INVALID_ARG;
    if (ws_bytes < lmhead_ws_bytes(M, K)) return QGEMV_WORKSPACE_TOO_SMALL;
    if (!aligned16(w_pack) || !aligned16(x) || !aligned16(cand) || !aligned16(ids) || !aligned16(top_vals) ||
        !aligned16(cand_vals) || !aligned16(workspace))
        return QGEMV_MISALIGNED;
    cudaStream_t s = as_stream(stream);
    // a candidate outside 0 .. N-1 keeps this NaN (all-ones bits)
    if (cudaMemsetAsync(cand_vals, 0xFF, (size_t)M * sizeof(float), s) != cudaSuccess) return QGEMV_CUDA_ERROR;
    uint8_t* xq = static_cast<uint8_t*>(workspace) + LMHEAD_Q8_OFFSET;
    st = launch_quantize_q8_1(x, ldx, xq, M, K, s);
    if (st != QGEMV_OK) return st;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.x = x;
    a.ldx = ldx;
    a.xq = xq;
    a.K = K;
    a.N = N;
    a.ws = static_cast<Top1Workspace*>(workspace);
    a.ids = ids;
    a.top_vals = top_vals;
    a.cand = cand;
    a.cand_vals = cand_vals;
    return launch_lmhead_q6_k(a, M, s);
}

int lmhead_q6_k_topk(const void* w_pack, const float* x, int64_t ldx, int k, const int32_t* cand, int32_t* ids,
                     float* vals, float* cand_vals, void* workspace, size_t ws_bytes, int M, int K, int N,
                     void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!w_pack || !x || !ids || !workspace || (cand == nullptr) != (cand_vals == nullptr)) return QGEMV_INVALID_ARG;
    int st = check_mk(M, K, QK_K);
    if (st) return st;
    if (N < 1 || ldx < K || k < 1 || k > QGEMV_TOPK_MAX || k > N) return QGEMV_INVALID_ARG;
    if (ws_bytes < topk_ws_bytes(M, K, N, k)) return QGEMV_WORKSPACE_TOO_SMALL;
    if (!aligned16(w_pack) || !aligned16(x) || !aligned16(ids) || !aligned16(workspace) || (vals && !aligned16(vals)) ||
        (cand && (!aligned16(cand) || !aligned16(cand_vals))))
        return QGEMV_MISALIGNED;
    cudaStream_t s = as_stream(stream);
    // a candidate outside 0 .. N-1 keeps this NaN (all-ones bits)
    if (cand && cudaMemsetAsync(cand_vals, 0xFF, (size_t)M * sizeof(float), s) != cudaSuccess) return QGEMV_CUDA_ERROR;
    uint8_t* xq = static_cast<uint8_t*>(workspace) + LMHEAD_Q8_OFFSET;
    st = launch_quantize_q8_1(x, ldx, xq, M, K, s);
    if (st != QGEMV_OK) return st;
    MmvqArgs a{};
    a.w_pack = w_pack;
    a.x = x;
    a.ldx = ldx;
    a.xq = xq;
    a.K = K;
    a.N = N;
    a.ws = static_cast<Top1Workspace*>(workspace);
    a.ids = ids;
    a.top_vals = vals;
    a.cand = cand;
    a.cand_vals = cand_vals;
    a.topk = k;
    a.topk_lists = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) + topk_lists_offset(M, K));
    return launch_lmhead_q6_k_topk(a, M, s);
}

int argmax_f32_rows(const float* y, int64_t ldy, int32_t* ids, void* workspace, size_t ws_bytes, int M, int N,
                    void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    if (!y || !ids || !workspace) return QGEMV_INVALID_ARG;
    if (M < 1 || N < 1 || ldy < N) return QGEMV_INVALID_ARG;
    if (M > QGEMV_MAX_M) return QGEMV_UNSUPPORTED_SHAPE;
    if (ws_bytes < top1_ws_bytes()) return QGEMV_WORKSPACE_TOO_SMALL;
    if (!aligned16(y) || !aligned16(ids) || !aligned16(workspace)) return QGEMV_MISALIGNED;
    return launch_argmax_rows(y, ldy, ids, static_cast<Top1Workspace*>(workspace), M, N, as_stream(stream));
}

int qgemv_block_dots_q4_0(const void* w_pack, const void* xq, int32_t* out, int M, int K, int N, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    int st = check_gemv(w_pack, xq, out, N, M, K, N, QK);
    if (st) return st;
    return launch_block_dots(FMT_Q4_0, w_pack, xq, out, M, K, N, as_stream(stream));
}

int qgemv_block_dots_q6_k(const void* w_pack, const void* xq, int32_t* out, int M, int K, int N, void* stream)
{
    QGEMV_FAIL_IF_TIMED_OUT();
    int st = check_gemv(w_pack, xq, out, N, M, K, N, QK_K);
    if (st) return st;
    return launch_block_dots(FMT_Q6_K, w_pack, xq, out, M, K, N, as_stream(stream));
}

int qgemv_set_q4_0_tensor_cores(int enable) { return set_q4_0_tensor_cores(enable); }

int qgemv_q4_0_plan(int M, int K, int N, int N_b, int* info)
{
    if (!info || M < 1 || K < QK || N < 1 || N_b < 0) return QGEMV_INVALID_ARG;
    if (M > QGEMV_MAX_M || K % QK) return QGEMV_UNSUPPORTED_SHAPE;
    for (int i = 0; i < 4; ++i) info[i] = 0;
    MmvqArgs a{};
    a.K = K;
    a.N = N;
    a.N2 = N_b;
    const int st = launch_mmvq_q4_0_tc(a, M, N_b > 0, nullptr, info);
    return st == TC_NOT_TAKEN ? QGEMV_OK : st;
}

int lmhead_q6_k_top1_plan(int M, int K, int N, int* info)
{
    if (!info || M < 1 || K < QK_K || N < 1) return QGEMV_INVALID_ARG;
    if (M > QGEMV_MAX_M || K % QK_K) return QGEMV_UNSUPPORTED_SHAPE;
    return lmhead_q6_k_plan(M, K, N, info);
}

int qgemv_set_q6_k_tensor_cores(int mode) { return set_q6_k_tensor_cores(mode); }

int qgemv_q6_k_plan(int M, int K, int N, int* info)
{
    if (!info || M < 1 || K < QK_K || N < 1) return QGEMV_INVALID_ARG;
    if (M > QGEMV_MAX_M || K % QK_K) return QGEMV_UNSUPPORTED_SHAPE;
    for (int i = 0; i < 4; ++i) info[i] = 0;
    MmvqArgs a{};
    a.K = K;
    a.N = N;
    const int st = launch_mmvq_q6_k_tc(a, M, nullptr, info);
    return st == TC_NOT_TAKEN ? QGEMV_OK : st;
}

int qgemv_q4_k_plan(int M, int K, int N, int* info)
{
    if (!info || M < 1 || K < QK_K || N < 1) return QGEMV_INVALID_ARG;
    if (M > QGEMV_MAX_M || K % QK_K) return QGEMV_UNSUPPORTED_SHAPE;
    for (int i = 0; i < 5; ++i) info[i] = 0;
    MmvqArgs a{};
    a.K = K;
    a.N = N;
    return launch_mmvq_q4_k(a, M, nullptr, info);
}

int qgemv_q5_k_plan(int M, int K, int N, int* info)
{
    if (!info || M < 1 || K < QK_K || N < 1) return QGEMV_INVALID_ARG;
    if (M > QGEMV_MAX_M || K % QK_K) return QGEMV_UNSUPPORTED_SHAPE;
    for (int i = 0; i < 5; ++i) info[i] = 0;
    MmvqArgs a{};
    a.K = K;
    a.N = N;
    return launch_mmvq_q5_k(a, M, nullptr, info);
}

int qgemv_q8_0_plan(int M, int K, int N, int* info)
{
    if (!info || M < 1 || K < QK || N < 1) return QGEMV_INVALID_ARG;
    if (M > QGEMV_MAX_M || K % (QK * 8)) return QGEMV_UNSUPPORTED_SHAPE;
    for (int i = 0; i < 5; ++i) info[i] = 0;
    MmvqArgs a{};
    a.K = K;
    a.N = N;
    return launch_mmvq_q8_0(a, M, nullptr, info);
}

int qgemv_take_wait_timeouts(unsigned int* count)
{
    if (!count) return QGEMV_INVALID_ARG;
    *count = 0;
    if (!wait_timeout_counter()) return QGEMV_CUDA_ERROR;
    if (g_counter_mapped) {
        *count = __atomic_exchange_n(&g_status_page[0], 0u, __ATOMIC_ACQ_REL);
        return QGEMV_OK;
    }
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_dev_counter, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_dev_counter, &zero, sizeof(zero)) != cudaSuccess)
        return QGEMV_CUDA_ERROR;
    *count = v;
    return QGEMV_OK;
}

int qgemv_debug_drop_next_copy(void) { return g_drop_request.exchange(1); }

int qgemv_bounds_check_build(void)
{
#ifdef QGEMV_BOUNDS_CHECK
    return 1;
#else
    return 0;
#endif
}

int qgemv_take_bounds_errors(unsigned int* count, unsigned int* first_site)
{
    if (!count || !first_site) return QGEMV_INVALID_ARG;
    *count = 0;
    *first_site = 0;
    if (!wait_timeout_counter()) return QGEMV_CUDA_ERROR;
    if (cudaDeviceSynchronize() != cudaSuccess) return QGEMV_CUDA_ERROR;
    if (g_counter_mapped) {
        *count = __atomic_exchange_n(&g_status_page[1], 0u, __ATOMIC_ACQ_REL);
        *first_site = __atomic_exchange_n(&g_status_page[2], 0u, __ATOMIC_ACQ_REL);
        return QGEMV_OK;
    }
    unsigned int v[3] = {0, 0, 0}, zero[2] = {0, 0};
    if (cudaMemcpyFromSymbol(v, g_dev_counter, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_dev_counter, zero, sizeof(zero), sizeof(unsigned int)) != cudaSuccess)
        return QGEMV_CUDA_ERROR;
    *count = v[1];
    *first_site = v[2];
    return QGEMV_OK;
}

int qgemv_debug_plant_bad_store(void)
{
#ifdef QGEMV_BOUNDS_CHECK
    return g_plant_request.exchange(1);
#else
    return QGEMV_UNSUPPORTED_SHAPE;
#endif
}

int qgemv_debug_fail_fused(int count) { return g_fail_fused.exchange(count > 0 ? count : 0); }

}  // extern "C"

namespace qgemv {

unsigned int* wait_timeout_counter()
{
    std::call_once(g_counter_once, counter_setup);
    return g_counter_dev;
}

bool wait_timeouts_pending() { return timeouts_pending(); }

int take_drop_request() { return g_drop_request.exchange(0); }

int take_plant_request() { return g_plant_request.exchange(0); }

}  // namespace qgemv
