// Small-M block-quantized matrix-vector kernels (Q4_0 / Q6_K weights against
// Q8_1 activations), plus the fused LM-head top-1 variant.
//
// What is computed (per output row n and activation row m):
//     y[m][n] = sum_b fp16(d_w[n,b]) * fp16(d_a[m,b]) * I[m,n,b]
// where I is the exact integer dot of block b ("Qwen3.6 27B Q4_0 DFlash/SYCL
// closure", What materially worked, item 2: direct Q4_0 MMVQ for rows 1-17;
// "Q6_K M=6 fused DFlash top-1 production record", Why this was slow: the
// five-row kernel reuses each weight slice across all rows).
//
// Work decomposition (GB300: 152 SMs, one CTA of up to 16 warps per SM):
//   * the N rows are split into groups of R rows; each CTA takes a contiguous,
//     balanced range of groups and its warps take the groups in turn;
//   * a warp walks its groups' (row, 32-block chunk) tiles in order and keeps
//     them streaming through a private ring of shared-memory stages filled by
//     TMA bulk copies (cp.async.bulk, completion on an mbarrier), several
//     stages ahead, so the bytes in flight do not depend on registers;
//   * lane l handles block l of every chunk for all R rows; it reuses one
//     activation block (staged once per CTA in shared memory) for R rows and
//     one weight block for M rows, holding R x M fp32 partial sums;
//   * a transpose-reduction sums the partials over the 32 lanes with the same
//     butterfly tree for every output, so an output's value does not depend on
//     where its row sits (duplicated rows give identical floats).
// Every weight byte is read from HBM once.  When the activation tile does not
// fit next to the rings (M * K large), a lock-step variant stages K in chunks
// and reads the weights with streaming loads (same arithmetic, same order).
#pragma once

#include "qgemv_common.cuh"

namespace qgemv {

constexpr int MMVQ_MAX_THREADS = 512;
constexpr int MMVQ_MAX_WARPS = MMVQ_MAX_THREADS / 32;

// Threads per CTA: 16 warps while the R x M partial sums are few; 8 warps
// (and so up to 255 registers per thread) for M > 8.
template <int M>
struct MmvqThreads {
    static constexpr int value = M <= 8 ? 512 : 256;
};

// Rows per warp: one 4-row group of the packed layout.
constexpr int R_ROWS = GROUP;

constexpr int next_pow2(int v) { return v <= 1 ? 1 : 2 * next_pow2((v + 1) / 2); }
constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// Sum P values (P a power of two) over the 32 lanes of a warp.  Afterwards a
// lane holds C = max(P / 32, 1) totals in a[0..C):
//   P >= 32: lane l holds values l * C + j;
//   P <  32: lane l holds value l >> (5 - log2 P) (32 / P lanes hold each).
// Every value is summed with the same pairing order (lanes 16 apart first,
// then 8, 4, 2, 1).
template <int P>
__device__ __forceinline__ void warp_transpose_reduce(float (&a)[P], int lane)
{
#pragma unroll
    for (int lvl = 0; lvl < 5; ++lvl) {
        const int off = 16 >> lvl;
        const int c = P >> lvl;
        if (c >= 2) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < c / 2; ++i) {
                float send = upper ? a[i] : a[i + c / 2];
                float keep = upper ? a[i + c / 2] : a[i];
                a[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        } else {
            a[0] += __shfl_xor_sync(0xffffffffu, a[0], off);
        }
    }
}

template <int P>
__device__ __forceinline__ int reduced_value_index(int lane, int j)
{
    if constexpr (P >= 32) return lane * (P / 32) + j;
    else return lane >> (5 - ilog2(P));
}

template <int P>
__device__ __forceinline__ bool reduced_value_owner(int lane)
{
    if constexpr (P >= 32) return true;
    else return (lane & ((32 / P) - 1)) == 0;
}

// ---------------------------------------------------------------------------
// TMA bulk copies and mbarriers (inline PTX).
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier shared-memory accesses before later TMA writes.
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for an mbarrier phase, giving up after about a second (returns false).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 1000000000ull) return false;
    }
    return true;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completing `bytes` of transaction on `bar`; weights are streamed once, so
// they are marked evict-first in L2.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// ---------------------------------------------------------------------------
// Activation staging into the shared tile.
// ---------------------------------------------------------------------------

struct ActTile {
    uint4* aq;  // [M][2][KC]
    uint2* am;  // [M][KC]
    int KC;
};

// From caller-supplied Q8_1 blocks in global memory.
template <int FMT, int M>
__device__ __forceinline__ void stage_from_q8_1(const ActTile& t, const uint8_t* xq, int NB, int kb0, int kb1)
{
    const int nbc = kb1 - kb0;
    for (int i = threadIdx.x; i < M * nbc; i += blockDim.x) {
        const int m = i / nbc, bl = i - m * nbc;
        uint4 lo, hi;
        uint2 meta;
        act_from_q8_1<FMT>(xq + ((int64_t)m * NB + kb0 + bl) * Q8_1_BYTES, lo, hi, meta);
        t.aq[(m * 2 + 0) * t.KC + bl] = lo;
        t.aq[(m * 2 + 1) * t.KC + bl] = hi;
        t.am[m * t.KC + bl] = meta;
    }
}

// From fp32 activations, quantizing to Q8_1 on the fly (one thread per block),
// bit-identical to the standalone quantize_q8_1 kernel.
template <int FMT, int M>
__device__ __forceinline__ void stage_from_f32(const ActTile& t, const float* x, int64_t ldx, int kb0, int kb1)
{
    const int nbc = kb1 - kb0;
    const bool vec4 = ((reinterpret_cast<uintptr_t>(x) | ((uintptr_t)ldx * 4)) & 15u) == 0;
    for (int i = threadIdx.x; i < M * nbc; i += blockDim.x) {
        const int m = i / nbc, bl = i - m * nbc;
        Q81Block qb;
        q8_1_quantize_block(x + (int64_t)m * ldx + (int64_t)(kb0 + bl) * QK, vec4, qb);
        t.aq[(m * 2 + 0) * t.KC + bl] = make_uint4(qb.q[0], qb.q[1], qb.q[2], qb.q[3]);
        t.aq[(m * 2 + 1) * t.KC + bl] = make_uint4(qb.q[4], qb.q[5], qb.q[6], qb.q[7]);
        uint2 meta;
        meta.x = __float_as_uint(__half2float(__float2half_rn(qb.d)));
        meta.y = act_meta_from_sums<FMT>(qb.s_lo, qb.s_hi);
        t.am[m * t.KC + bl] = meta;
    }
}

// ---------------------------------------------------------------------------
// Per-block accumulation, shared by both kernel variants.
// ---------------------------------------------------------------------------

// Q4_0: w16[r] = the block's 16 code bytes of row r, dw[r] = its scale.
template <int M, int R>
__device__ __forceinline__ void accumulate_q4_0(const uint4 (&w16)[R], const float (&dw)[R], const ActTile& t, int ti,
                                                float (&acc)[R][M])
{
    uint32_t w[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) q4_0_unpack(w16[r], w[r]);
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 lo = t.aq[(m * 2 + 0) * t.KC + ti];
        const uint4 hi = t.aq[(m * 2 + 1) * t.KC + ti];
        const uint2 mt = t.am[m * t.KC + ti];
        const float da = __uint_as_float(mt.x);
        const int init = (int)mt.y + MAGIC_I2F_BITS;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int s = q4_0_dot(w[r], lo, hi, init);
            const float f = __int_as_float(s) - MAGIC_I2F;  // exact I
            acc[r][m] = fmaf(dw[r] * da, f, acc[r][m]);
        }
    }
}

// Q6_K: ql/qh/sc of the block for row r, dw[r] = its superblock scale.
template <int M, int R>
__device__ __forceinline__ void accumulate_q6_k(const uint4 (&ql)[R], const uint2 (&qh)[R], const uint32_t (&sc)[R],
                                                const float (&dw)[R], const ActTile& t, int ti, float (&acc)[R][M])
{
    uint32_t w[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) q6_k_unpack(ql[r], qh[r], w[r]);
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 lo = t.aq[(m * 2 + 0) * t.KC + ti];
        const uint4 hi = t.aq[(m * 2 + 1) * t.KC + ti];
        const uint2 mt = t.am[m * t.KC + ti];
        const float da = __uint_as_float(mt.x);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int J = q6_k_dot(w[r], lo, hi, mt.y, sc[r]);
            acc[r][m] = fmaf(dw[r] * da, (float)J, acc[r][m]);
        }
    }
}

// ---------------------------------------------------------------------------
// Block-major activation tile of the Q6_K ring kernel: for block b the codes
// of rows m = 0..M-1 lie at ab[b] + 32 m (two 16-byte halves), with a block
// stride of (2M + 1) * 16 bytes (an odd number of 16-byte units, so that the
// 32 lanes, which read 32 consecutive blocks, hit distinct bank groups), and
// the per-(block, row) meta word at am[b * M + m].  One base address per lane
// and compile-time offsets per row m.
// ---------------------------------------------------------------------------

template <int M>
struct BlockAct {
    static constexpr int STRIDE = (2 * M + 1) * 16;
    uint8_t* q;  // [NB][STRIDE]
    uint2* am;   // [NB][M]
};

template <int FMT, int M>
__device__ __forceinline__ void block_act_from_q8_1(const BlockAct<M>& t, const uint8_t* xq, int NB)
{
    for (int i = threadIdx.x; i < M * NB; i += blockDim.x) {
        const int m = i / NB, b = i - m * NB;
        uint4 lo, hi;
        uint2 meta;
        act_from_q8_1<FMT>(xq + ((int64_t)m * NB + b) * Q8_1_BYTES, lo, hi, meta);
        uint4* dst = reinterpret_cast<uint4*>(t.q + b * BlockAct<M>::STRIDE + 32 * m);
        dst[0] = lo;
        dst[1] = hi;
        t.am[b * M + m] = meta;
    }
}

template <int FMT, int M>
__device__ __forceinline__ void block_act_from_f32(const BlockAct<M>& t, const float* x, int64_t ldx, int NB)
{
    const bool vec4 = ((reinterpret_cast<uintptr_t>(x) | ((uintptr_t)ldx * 4)) & 15u) == 0;
    for (int i = threadIdx.x; i < M * NB; i += blockDim.x) {
        const int m = i / NB, b = i - m * NB;
        Q81Block qb;
        q8_1_quantize_block(x + (int64_t)m * ldx + (int64_t)b * QK, vec4, qb);
        uint4* dst = reinterpret_cast<uint4*>(t.q + b * BlockAct<M>::STRIDE + 32 * m);
        dst[0] = make_uint4(qb.q[0], qb.q[1], qb.q[2], qb.q[3]);
        dst[1] = make_uint4(qb.q[4], qb.q[5], qb.q[6], qb.q[7]);
        uint2 meta;
        meta.x = __float_as_uint(__half2float(__float2half_rn(qb.d)));
        meta.y = act_meta_from_sums<FMT>(qb.s_lo, qb.s_hi);
        t.am[b * M + m] = meta;
    }
}

// Q4_0 block of R rows against the block-major tile (block index ti).
template <int M, int R>
__device__ __forceinline__ void accumulate_q4_0_blk(const uint4 (&w16)[R], const float (&dw)[R],
                                                    const BlockAct<M>& t, int ti, float (&acc)[R][M])
{
    uint32_t w[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) q4_0_unpack(w16[r], w[r]);
    const uint8_t* ab = t.q + ti * BlockAct<M>::STRIDE;
    const uint2* am = t.am + ti * M;
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 lo = *reinterpret_cast<const uint4*>(ab + 32 * m);
        const uint4 hi = *reinterpret_cast<const uint4*>(ab + 32 * m + 16);
        const uint2 mt = am[m];
        const float da = __uint_as_float(mt.x);
        const int init = (int)mt.y + MAGIC_I2F_BITS;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int sI = q4_0_dot(w[r], lo, hi, init);
            const float f = __int_as_float(sI) - MAGIC_I2F;  // exact I
            acc[r][m] = fmaf(dw[r] * da, f, acc[r][m]);
        }
    }
}

// Q6_K block of R rows against the block-major tile (block index ti).
template <int M, int R>
__device__ __forceinline__ void accumulate_q6_k_blk(const uint4 (&ql)[R], const uint2 (&qh)[R],
                                                    const uint32_t (&sc)[R], const float (&dw)[R],
                                                    const BlockAct<M>& t, int ti, float (&acc)[R][M])
{
    uint32_t w[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) q6_k_unpack(ql[r], qh[r], w[r]);
    const uint8_t* ab = t.q + ti * BlockAct<M>::STRIDE;
    const uint2* am = t.am + ti * M;
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 lo = *reinterpret_cast<const uint4*>(ab + 32 * m);
        const uint4 hi = *reinterpret_cast<const uint4*>(ab + 32 * m + 16);
        const uint2 mt = am[m];
        const float da = __uint_as_float(mt.x);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int J = q6_k_dot(w[r], lo, hi, mt.y, sc[r]);
            acc[r][m] = fmaf(dw[r] * da, (float)J, acc[r][m]);
        }
    }
}

// ---------------------------------------------------------------------------
// Kernel arguments and epilogue.
// ---------------------------------------------------------------------------

struct MmvqArgs {
    const void* w_pack;
    const uint8_t* xq;  // Q8_1 [M][NB] (TOP1 = false)
    const float* x;     // fp32 [M][ldx] (TOP1 = true)
    int64_t ldx;
    float* y;
    int64_t ldy;
    int K, N;
    int KC;      // activation blocks staged at once (lock-step kernel)
    int stages;  // ring stages per warp (ring kernel)
    Top1Workspace* ws;
    int32_t* ids;
};

// Reduce one row group's partial sums over the warp and write them (TOP1 =
// false) or fold their keys into the warp's running best per row (TOP1).
template <int M, int R, bool TOP1>
__device__ __forceinline__ void finish_rowgroup(const MmvqArgs& a, int n0, float (&acc)[R][M], int lane,
                                                unsigned long long* wk, unsigned long long& best)
{
    constexpr int V = R * M;
    constexpr int P = next_pow2(V);
    constexpr int C = P >= 32 ? P / 32 : 1;
    float v[P];
#pragma unroll
    for (int i = 0; i < P; ++i) v[i] = i < V ? acc[i / M][i % M] : 0.0f;
    warp_transpose_reduce<P>(v, lane);
    if (!TOP1) {
        if (reduced_value_owner<P>(lane)) {
#pragma unroll
            for (int j = 0; j < C; ++j) {
                const int vi = reduced_value_index<P>(lane, j);
                if (vi < V) {
                    const int r = vi / M, m = vi - (vi / M) * M;
                    const int n = n0 + r;
                    if (n < a.N) a.y[(int64_t)m * a.ldy + n] = v[j];
                }
            }
        }
    } else {
        if (reduced_value_owner<P>(lane)) {
#pragma unroll
            for (int j = 0; j < C; ++j) {
                const int vi = reduced_value_index<P>(lane, j);
                if (vi < V) {
                    const int n = n0 + vi / M;
                    wk[vi] = n < a.N ? top1_key(v[j], n) : 0ull;
                }
            }
        }
        __syncwarp();
        if (lane < M) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const unsigned long long k = wk[r * M + lane];
                best = k > best ? k : best;
            }
        }
        __syncwarp();
    }
}

// Combine the warps' best keys, then across CTAs with one 64-bit atomicMax per
// row; the last CTA to finish writes the ids and leaves the workspace zeroed.
template <int M>
__device__ __forceinline__ void top1_finish(const MmvqArgs& a, unsigned long long* s_best, int* s_last,
                                            unsigned long long best, int lane, int warp, int nwarps)
{
    if (lane < M) s_best[warp * MAX_M + lane] = best;
    __syncthreads();
    if (threadIdx.x < M) {
        unsigned long long k = 0ull;
        for (int w = 0; w < nwarps; ++w) {
            const unsigned long long kw = s_best[w * MAX_M + threadIdx.x];
            k = kw > k ? kw : k;
        }
        atomicMax(&a.ws->keys[threadIdx.x], k);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&a.ws->done, 1u);
        *s_last = prev == gridDim.x - 1;
    }
    __syncthreads();
    if (*s_last) {
        __threadfence();
        if (threadIdx.x < M) {
            const unsigned long long k = atomicExch(&a.ws->keys[threadIdx.x], 0ull);
            a.ids[threadIdx.x] = top1_key_to_id(k);
        }
        if (threadIdx.x == 0) atomicExch(&a.ws->done, 0u);
    }
}

// Shared memory besides the activation tile and the rings, for TOP1.
inline size_t top1_scratch_bytes(int nwarps) { return (size_t)nwarps * 64 * 8 + (size_t)nwarps * MAX_M * 8 + 16; }

// ---------------------------------------------------------------------------
// Ring kernel: the whole activation in shared memory, weights streamed by
// per-warp TMA rings.
//   shared memory: rings [W][S][stage] | aq [M][2][NB] | am [M][NB] |
//                  mbarriers [W][S] | TOP1 scratch
// The CTA's groups are g0 .. g1-1; warp w takes g0 + w, g0 + w + W, ...
// Job j of a warp = (its group j / nch, chunk j % nch), in stage j % S: one
// bulk copy of the group-chunk (4 rows' tiles and, for Q6_K, their scales).
// Waits are bounded: a warp that waits about a second for a copy counts a
// timeout in *timeouts, stops, and gives its copies in flight a bounded wait.
// ---------------------------------------------------------------------------

template <int FMT, int M, bool TOP1>
__global__ void __launch_bounds__(MmvqThreads<M>::value, 1) mmvq_ring_kernel(const MmvqArgs a, unsigned int* timeouts)
{
    constexpr int R = R_ROWS;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
    const int S = a.stages;
    const Layout L = make_layout(FMT, a.N, a.K);
    const int NB = L.NB, nch = L.nch;
    const int stage_bytes = L.chunk_bytes(R, 0);

    uint8_t* rings = smem;
    BlockAct<M> t;
    t.q = rings + (size_t)W * S * stage_bytes;
    t.am = reinterpret_cast<uint2*>(t.q + (size_t)NB * BlockAct<M>::STRIDE);
    uint64_t* bars = reinterpret_cast<uint64_t*>(t.am + M * NB);
    unsigned long long* s_keys = reinterpret_cast<unsigned long long*>(bars + W * S);  // [W][64]
    unsigned long long* s_best = s_keys + W * 64;                                     // [W][MAX_M]
    int* s_last = reinterpret_cast<int*>(s_best + W * MAX_M);

    const int64_t g0 = (int64_t)blockIdx.x * L.n_groups / gridDim.x;
    const int64_t g1 = (int64_t)(blockIdx.x + 1) * L.n_groups / gridDim.x;
    const int n_my = warp < g1 - g0 ? (int)((g1 - g0 - warp + W - 1) / W) : 0;
    const int J = n_my * nch;

    uint64_t* wbar = bars + warp * S;
    uint8_t* wring = rings + (size_t)warp * S * stage_bytes;
    const uint8_t* wbase = static_cast<const uint8_t*>(a.w_pack);
    const uint64_t pol = l2_evict_first_policy();

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&wbar[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    // Issue cursor (lane 0): next job's group, chunk and stage.
    int issued = 0, iss_c = 0, iss_slot = 0;
    int64_t iss_g = g0 + warp;
    const int64_t GB = L.group_bytes(GROUP);  // bytes of a full group
    const int CB = L.chunk_bytes(GROUP, 0);    // bytes of a full chunk of a full group
    auto issue_next = [&]() {
        const int rows = L.rows_in(iss_g);
        const bool full = rows == GROUP && (iss_c < nch - 1 || L.nb_tail == CHUNK);
        const uint32_t bytes = full ? (uint32_t)CB : (uint32_t)L.chunk_bytes(rows, iss_c);
        const int64_t off = iss_g * GB + (int64_t)iss_c * (rows == GROUP ? CB : L.chunk_bytes(rows, 0));
        uint64_t* bar = &wbar[iss_slot];
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(wring + (size_t)iss_slot * stage_bytes, wbase + off, bytes, bar, pol);
        ++issued;
        if (++iss_slot == S) iss_slot = 0;
        if (++iss_c == nch) {
            iss_c = 0;
            iss_g += W;
        }
    };
    if (lane == 0) {
        while (issued < S - 1 && issued < J) issue_next();
    }

    // The activation is staged while the first weight tiles are in flight.
    if (TOP1) block_act_from_f32<FMT, M>(t, a.x, a.ldx, NB);
    else block_act_from_q8_1<FMT, M>(t, a.xq, NB);
    __syncthreads();

    unsigned long long best = 0ull;
    float acc[R][M];
    int consumed = 0;
    int c = 0, slot = 0;
    uint32_t phase = 0;
    int64_t g = g0 + warp;
    for (int j = 0; j < J; ++j) {
        if (lane == 0 && issued < J) {
            fence_proxy_async();
            issue_next();
        }
        if (c == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;
        }
        const bool ready = __all_sync(0xffffffffu, mbar_wait_bounded(&wbar[slot], phase));
        if (!ready) {
            if (lane == 0) atomicAdd(timeouts, 1u);
            break;
        }
        consumed = j + 1;
        const uint8_t* st = wring + (size_t)slot * stage_bytes;
        const int rows = L.rows_in(g);
        const int ti = c * CHUNK + lane;
        const bool full_chunk = c != nch - 1 || L.nb_tail == CHUNK;
        if (FMT == FMT_Q4_0) {
            // block-major group-chunk: nib[block][row] then d[block][row]
            uint4 w16[R];
            float dw[R];
            if (full_chunk && rows == R) {
#pragma unroll
                for (int r = 0; r < R; ++r) w16[r] = *reinterpret_cast<const uint4*>(st + (lane * R + r) * 16);
                const uint2 dd = *reinterpret_cast<const uint2*>(st + CHUNK * R * 16 + lane * R * 2);
                dw[0] = __half2float(__ushort_as_half((unsigned short)(dd.x & 0xFFFFu)));
                dw[1] = __half2float(__ushort_as_half((unsigned short)(dd.x >> 16)));
                dw[2] = __half2float(__ushort_as_half((unsigned short)(dd.y & 0xFFFFu)));
                dw[3] = __half2float(__ushort_as_half((unsigned short)(dd.y >> 16)));
                accumulate_q4_0_blk<M, R>(w16, dw, t, ti, acc);
            } else if (lane < L.nb(c)) {
                // rows past the group's end read stale data; their sums are discarded
                const int nb = L.nb(c);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int rr = min(r, rows - 1);
                    w16[r] = *reinterpret_cast<const uint4*>(st + (lane * rows + rr) * 16);
                    dw[r] = __half2float(__ushort_as_half(
                        *reinterpret_cast<const uint16_t*>(st + nb * rows * 16 + (lane * rows + rr) * 2)));
                }
                accumulate_q4_0_blk<M, R>(w16, dw, t, ti, acc);
            }
        } else {
        uint4 ql[R];
        uint2 qh[R];
        uint32_t sc[R];
        float dw[R];
        if (full_chunk) {
            if (rows == R) {
                // full chunk of a full group: every offset is a compile-time constant
                constexpr int TB = CHUNK * 26;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    ql[r] = *reinterpret_cast<const uint4*>(st + r * TB + lane * 16);
                    qh[r] = *reinterpret_cast<const uint2*>(st + r * TB + CHUNK * 16 + lane * 8);
                    sc[r] = *reinterpret_cast<const uint16_t*>(st + r * TB + CHUNK * 24 + lane * 2);
                    dw[r] = __half2float(__ushort_as_half(
                        *reinterpret_cast<const uint16_t*>(st + R * TB + (r * (CHUNK / 8) + (lane >> 3)) * 2)));
                }
            } else {
                constexpr int TB = CHUNK * 26;
                const uint16_t* dq = reinterpret_cast<const uint16_t*>(st + rows * TB);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    // rows past the group's end read stale data; their sums are discarded
                    ql[r] = *reinterpret_cast<const uint4*>(st + r * TB + lane * 16);
                    qh[r] = *reinterpret_cast<const uint2*>(st + r * TB + CHUNK * 16 + lane * 8);
                    sc[r] = *reinterpret_cast<const uint16_t*>(st + r * TB + CHUNK * 24 + lane * 2);
                    dw[r] = __half2float(__ushort_as_half(dq[min(r, rows - 1) * (CHUNK / 8) + (lane >> 3)]));
                }
            }
            accumulate_q6_k_blk<M, R>(ql, qh, sc, dw, t, ti, acc);
        } else if (lane < L.nb_tail) {
            const int nb = L.nb_tail, tb = nb * 26;
            const uint16_t* dq = reinterpret_cast<const uint16_t*>(st + rows * tb);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                ql[r] = *reinterpret_cast<const uint4*>(st + r * tb + lane * 16);
                qh[r] = *reinterpret_cast<const uint2*>(st + r * tb + nb * 16 + lane * 8);
                sc[r] = *reinterpret_cast<const uint16_t*>(st + r * tb + nb * 24 + lane * 2);
                dw[r] = __half2float(__ushort_as_half(dq[min(r, rows - 1) * (nb >> 3) + (lane >> 3)]));
            }
            accumulate_q6_k_blk<M, R>(ql, qh, sc, dw, t, ti, acc);
        }
        }
        __syncwarp();
        if (c == nch - 1) finish_rowgroup<M, R, TOP1>(a, (int)(g * GROUP), acc, lane, s_keys + warp * 64, best);
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
        if (++c == nch) {
            c = 0;
            g += W;
        }
    }
    // After a timeout, give the copies still in flight a bounded wait before
    // the shared memory is released.
    if (lane == 0) {
        for (int jj = consumed; jj < issued; ++jj) mbar_wait_bounded(&wbar[jj % S], (uint32_t)((jj / S) & 1));
    }
    __syncwarp();

    if (TOP1) top1_finish<M>(a, s_best, s_last, best, lane, warp, W);
}

// ---------------------------------------------------------------------------
// Lock-step kernel: for activations too large for shared memory next to the
// rings.  K is staged in chunks of KC blocks (a multiple of 32); all warps
// move through the chunks together; weights are read with streaming loads.
//   shared memory: aq [M][2][KC] | am [M][KC] | TOP1 scratch
// ---------------------------------------------------------------------------

template <int FMT, int M, bool TOP1>
__global__ void __launch_bounds__(MmvqThreads<M>::value, 1) mmvq_lockstep_kernel(const MmvqArgs a)
{
    constexpr int R = R_ROWS;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
    const Layout L = make_layout(FMT, a.N, a.K);
    const int NB = L.NB, KC = a.KC;
    ActTile t;
    t.aq = reinterpret_cast<uint4*>(smem);
    t.am = reinterpret_cast<uint2*>(t.aq + 2 * M * KC);
    t.KC = KC;
    unsigned long long* s_keys = reinterpret_cast<unsigned long long*>(t.am + M * KC);
    unsigned long long* s_best = s_keys + W * 64;
    int* s_last = reinterpret_cast<int*>(s_best + W * MAX_M);

    const int64_t n_items = (L.n_groups + W - 1) / W;
    const int nchunks = (NB + KC - 1) / KC;
    unsigned long long best = 0ull;

    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int64_t g = item * W + warp;
        const bool active = g < L.n_groups;
        int rows[R];
#pragma unroll
        for (int r = 0; r < R; ++r) rows[r] = (int)min(g * GROUP + r, (int64_t)a.N - 1);
        float acc[R][M];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;
        for (int cc = 0; cc < nchunks; ++cc) {
            const int kb0 = cc * KC, kb1 = min(NB, kb0 + KC);
            __syncthreads();
            if (TOP1) stage_from_f32<FMT, M>(t, a.x, a.ldx, kb0, kb1);
            else stage_from_q8_1<FMT, M>(t, a.xq, NB, kb0, kb1);
            __syncthreads();
            if (!active) continue;
            for (int b = kb0 + lane; b < kb1; b += 32) {
                const int ti = b - kb0;
                if (FMT == FMT_Q4_0) {
                    uint4 w16[R];
                    float dw[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const BlockAddr ad = block_addr(a.w_pack, L, rows[r], b);
                        w16[r] = ld_stream_v4(reinterpret_cast<const uint4*>(ad.q));
                        dw[r] = __half2float(__ushort_as_half(ld_stream_u16(ad.d)));
                    }
                    accumulate_q4_0<M, R>(w16, dw, t, ti, acc);
                } else {
                    uint4 ql[R];
                    uint2 qh[R];
                    uint32_t sc[R];
                    float dw[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const BlockAddr ad = block_addr(a.w_pack, L, rows[r], b);
                        ql[r] = ld_stream_v4(reinterpret_cast<const uint4*>(ad.q));
                        qh[r] = ld_stream_v2(reinterpret_cast<const uint2*>(ad.qh));
                        sc[r] = ld_stream_u16(ad.sc);
                        dw[r] = __half2float(__ushort_as_half(ld_stream_u16(ad.d)));
                    }
                    accumulate_q6_k<M, R>(ql, qh, sc, dw, t, ti, acc);
                }
            }
        }
        if (active) finish_rowgroup<M, R, TOP1>(a, (int)(g * GROUP), acc, lane, s_keys + warp * 64, best);
    }
    if (TOP1) top1_finish<M>(a, s_best, s_last, best, lane, warp, W);
}

}  // namespace qgemv
